// Row movement around the expert GEMMs.
//
// gather : Xp[r] = x[perm[r] / k] for the kept rows r < R = offsets[E] -- the tokens of each
//          expert laid out as one contiguous batch ("Mixture of experts (MoE)", tirogla.com,
//          How it works, step 4: each expert runs on its contiguous batch).
// combine: y[t] = sum over slots s < k with inv[t*k+s] >= 0 of Yp[inv[t*k+s]] (+ S[t]),
//          summed in slot order in fp32; a dropped assignment adds nothing (same page,
//          step 5). Yp already carries the gate (applied in the down-projection epilogue).
//
// Both are HBM-bound copies: one warp per row, 16-byte vector loads and stores, several
// loads in flight per lane, grid sized as a multiple of the SM count.
#include <algorithm>

#include "common.cuh"
#include "launchers.h"

namespace moe {

namespace {

constexpr int kMoveThreads = 256;
constexpr int kMoveWarps = kMoveThreads / 32;

__global__ void __launch_bounds__(kMoveThreads)
gather_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ perm,
                   const int32_t* __restrict__ offsets, int E, int k, int nvec,
                   uint4* __restrict__ xp) {
  const int R = offsets[E];
  const int lane = threadIdx.x & 31;
  const int nw = gridDim.x * kMoveWarps;
  for (int r = blockIdx.x * kMoveWarps + (threadIdx.x >> 5); r < R; r += nw) {
    const int t = perm[r] / k;
    const uint4* src = x + static_cast<size_t>(t) * nvec;
    uint4* dst = xp + static_cast<size_t>(r) * nvec;
    int i = lane;
    for (; i + 96 < nvec; i += 128) {
      const uint4 a = __ldg(src + i), b = __ldg(src + i + 32), c = __ldg(src + i + 64),
                  d = __ldg(src + i + 96);
      dst[i] = a;
      dst[i + 32] = b;
      dst[i + 64] = c;
      dst[i + 96] = d;
    }
    for (; i < nvec; i += 32) dst[i] = __ldg(src + i);
  }
}

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    acc[2 * q] += __uint_as_float(w[q] << 16);
    acc[2 * q + 1] += __uint_as_float(w[q] & 0xffff0000u);
  }
}

// One warp per token; each lane owns 16-byte chunks of the row (8 bf16 values).
__global__ void __launch_bounds__(kMoveThreads)
combine_bf16_kernel(const uint4* __restrict__ yp, const int32_t* __restrict__ inv,
                    const uint4* __restrict__ ys, uint4* __restrict__ y, int T, int k, int nvec) {
  const int lane = threadIdx.x & 31;
  const int nw = gridDim.x * kMoveWarps;
  for (int t = blockIdx.x * kMoveWarps + (threadIdx.x >> 5); t < T; t += nw) {
    const int32_t* slots = inv + static_cast<size_t>(t) * k;
    for (int i = lane; i < nvec; i += 32) {
      float acc[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = 0.f;
      for (int s = 0; s < k; ++s) {
        const int r = __ldg(slots + s);
        if (r >= 0) add_bf16x8(acc, __ldg(yp + static_cast<size_t>(r) * nvec + i));
      }
      if (ys != nullptr) add_bf16x8(acc, __ldg(ys + static_cast<size_t>(t) * nvec + i));
      y[static_cast<size_t>(t) * nvec + i] =
          make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                     pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    }
  }
}

// fp32 variant: 16-byte chunks of 4 floats.
__global__ void __launch_bounds__(kMoveThreads)
combine_f32_kernel(const float4* __restrict__ yp, const int32_t* __restrict__ inv,
                   const float4* __restrict__ ys, float4* __restrict__ y, int T, int k, int nvec) {
  const int lane = threadIdx.x & 31;
  const int nw = gridDim.x * kMoveWarps;
  for (int t = blockIdx.x * kMoveWarps + (threadIdx.x >> 5); t < T; t += nw) {
    const int32_t* slots = inv + static_cast<size_t>(t) * k;
    for (int i = lane; i < nvec; i += 32) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s = 0; s < k; ++s) {
        const int r = __ldg(slots + s);
        if (r >= 0) {
          const float4 v = __ldg(yp + static_cast<size_t>(r) * nvec + i);
          acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
      }
      if (ys != nullptr) {
        const float4 v = __ldg(ys + static_cast<size_t>(t) * nvec + i);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
      y[static_cast<size_t>(t) * nvec + i] = acc;
    }
  }
}

int grid_for_rows(long long rows, int num_sms) {
  const long long want = (rows + kMoveWarps - 1) / kMoveWarps;
  const long long cap = static_cast<long long>(std::max(num_sms, 1)) * 8;
  return static_cast<int>(std::max<long long>(1, std::min(want, cap)));
}

}  // namespace

int launch_gather(const void* x, const int32_t* perm, const int32_t* offsets, int E, int k,
                  int row_bytes, int max_rows, void* xp, int num_sms, cudaStream_t stream) {
  if (max_rows <= 0) return MOE_OK;
  gather_rows_kernel<<<grid_for_rows(max_rows, num_sms), kMoveThreads, 0, stream>>>(
      static_cast<const uint4*>(x), perm, offsets, E, k, row_bytes / 16, static_cast<uint4*>(xp));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_combine(int dtype, const void* yp, const int32_t* inv, const void* ys, void* y, int T,
                   int k, int d, int num_sms, cudaStream_t stream) {
  if (T <= 0) return MOE_OK;
  const int grid = grid_for_rows(T, num_sms);
  if (dtype == MOE_BF16) {
    combine_bf16_kernel<<<grid, kMoveThreads, 0, stream>>>(
        static_cast<const uint4*>(yp), inv, static_cast<const uint4*>(ys), static_cast<uint4*>(y),
        T, k, d / 8);
  } else {
    combine_f32_kernel<<<grid, kMoveThreads, 0, stream>>>(
        static_cast<const float4*>(yp), inv, static_cast<const float4*>(ys),
        static_cast<float4*>(y), T, k, d / 4);
  }
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
