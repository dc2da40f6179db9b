// Row movement around the expert GEMMs.
//
// gather : Xp[r] = x[perm[r] / k] for the kept rows r < R = offsets[E] -- the tokens of each
//          expert laid out as one contiguous batch ("Mixture of experts (MoE)", tirogla.com,
//          How it works, step 4: each expert runs on its contiguous batch). For top-1 layers
//          whose down projection writes y directly, a token-major form that also zeroes the
//          rows of dropped tokens (step 5 with k = 1 is a copy, which the GEMM's epilogue does).
// combine: y[t] = sum over slots s < k with inv[t*k+s] >= 0 of Yp[inv[t*k+s]] (+ S[t]),
//          summed in slot order in fp32; a dropped assignment adds nothing (same page,
//          step 5). Yp already carries the gate (applied in the down-projection epilogue).
//
// Both are HBM-bound copies: one warp per row (the combine: per 1 KB segment of a row),
// 16-byte vector loads and stores, every load of a row's piece issued before its stores,
// grid sized as a multiple of the SM count.
#include <algorithm>

#include "common.cuh"
#include "launchers.h"

namespace moe {

namespace {

constexpr int kMoveThreads = 256;
constexpr int kMoveWarps = kMoveThreads / 32;

// Copies one row of nvec 16-byte chunks with one warp: up to 16 chunks per lane are loaded
// before any is stored, so a row of up to 8 KB costs one memory round trip.
__device__ __forceinline__ void copy_row(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                         int nvec, int lane) {
  constexpr int U = 16;
  for (int i0 = 0; i0 < nvec; i0 += 32 * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + lane + 32 * u;
      if (i < nvec) v[u] = __ldg(src + i);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + lane + 32 * u;
      if (i < nvec) dst[i] = v[u];
    }
  }
}

__global__ void __launch_bounds__(kMoveThreads)
gather_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ perm,
                   const int32_t* __restrict__ offsets, int E, int k, int nvec,
                   uint4* __restrict__ xp) {
  pdl_wait();
  pdl_launch_dependents();
  const int R = offsets[E];
  const int lane = threadIdx.x & 31;
  const int nw = gridDim.x * kMoveWarps;
  for (int r = blockIdx.x * kMoveWarps + (threadIdx.x >> 5); r < R; r += nw) {
    const int t = perm[r] / k;
    copy_row(x + static_cast<size_t>(t) * nvec, xp + static_cast<size_t>(r) * nvec, nvec, lane);
  }
}

// Top-1 layers whose down projection writes y itself (its epilogue stores row r at token
// perm[r]): one warp per token t, Xp[inv[t]] = x[t] for a kept token, y[t] = 0 for a dropped
// one (the combine's result for a token with no kept assignment). Each y row is written
// exactly once between this kernel and the GEMM.
__global__ void __launch_bounds__(kMoveThreads)
gather_tokens_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ inv, int T,
                     int nvec, uint4* __restrict__ xp, uint4* __restrict__ y) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int nw = gridDim.x * kMoveWarps;
  for (int t = blockIdx.x * kMoveWarps + (threadIdx.x >> 5); t < T; t += nw) {
    const int r = __ldg(inv + t);
    if (r >= 0) {
      copy_row(x + static_cast<size_t>(t) * nvec, xp + static_cast<size_t>(r) * nvec, nvec, lane);
    } else {
      uint4* dst = y + static_cast<size_t>(t) * nvec;
      for (int i = lane; i < nvec; i += 32) dst[i] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// Gather with a bf16 -> fp16 conversion (operand of the 8-bit-weight GEMMs). A value outside
// fp16's finite range records MOE_ERR_NONFINITE (site SITE_F16_RANGE_X, detail = row).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w, bool& bad) {
  const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xffff0000u);
  bad |= fabsf(lo) > kF16Max || fabsf(hi) > kF16Max;
  return pack_f16x2(lo, hi);
}

__global__ void __launch_bounds__(kMoveThreads)
gather_rows_f16_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ perm,
                       const int32_t* __restrict__ offsets, int E, int k, int nvec,
                       uint4* __restrict__ xp, DeviceError* err) {
  pdl_wait();
  pdl_launch_dependents();
  const int R = offsets[E];
  const int lane = threadIdx.x & 31;
  const int nw = gridDim.x * kMoveWarps;
  for (int r = blockIdx.x * kMoveWarps + (threadIdx.x >> 5); r < R; r += nw) {
    const int t = perm[r] / k;
    const uint4* src = x + static_cast<size_t>(t) * nvec;
    uint4* dst = xp + static_cast<size_t>(r) * nvec;
    bool bad = false;
    for (int i = lane; i < nvec; i += 32) {
      const uint4 v = __ldg(src + i);
      dst[i] = make_uint4(bf16x2_to_f16x2(v.x, bad), bf16x2_to_f16x2(v.y, bad),
                          bf16x2_to_f16x2(v.z, bad), bf16x2_to_f16x2(v.w, bad));
    }
    if (bad) record_error(err, MOE_ERR_NONFINITE, SITE_F16_RANGE_X, r);
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

__device__ __forceinline__ void add_f32x4(float (&acc)[8], const uint4 v) {
  acc[0] += __uint_as_float(v.x);
  acc[1] += __uint_as_float(v.y);
  acc[2] += __uint_as_float(v.z);
  acc[3] += __uint_as_float(v.w);
}

template <bool BF16>
__device__ __forceinline__ void add_chunk(float (&acc)[8], const uint4 v) {
  if (BF16) add_bf16x8(acc, v); else add_f32x4(acc, v);
}

template <bool BF16>
__device__ __forceinline__ uint4 pack_chunk(const float (&acc)[8]) {
  if (BF16)
    return make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                      pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
  return make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]), __float_as_uint(acc[2]),
                    __float_as_uint(acc[3]));
}

// One warp per (token, segment of 64 16-byte chunks); each lane owns chunks c and c + 32 of
// the segment. KS > 0 unrolls the slot loop: all 2 * KS loads, and the shared expert's two,
// are issued before the first add (one memory round trip per task; more chunks per task left
// too few tasks for small batches). KS == 0 handles any k. Sums run in slot order in fp32,
// the shared expert last.
template <bool BF16, int KS>
__global__ void __launch_bounds__(kMoveThreads)
combine_kernel(const uint4* __restrict__ yp, const int32_t* __restrict__ inv,
               const uint4* __restrict__ ys, uint4* __restrict__ y, int T, int k, int nvec) {
  pdl_wait();
  pdl_launch_dependents();
  constexpr int CH = 2;
  const int lane = threadIdx.x & 31;
  const int nseg = (nvec + 32 * CH - 1) / (32 * CH);
  const long long total = static_cast<long long>(T) * nseg;
  const long long nw = static_cast<long long>(gridDim.x) * kMoveWarps;
  for (long long w = static_cast<long long>(blockIdx.x) * kMoveWarps + (threadIdx.x >> 5); w < total;
       w += nw) {
    const int t = static_cast<int>(w / nseg);
    const int seg = static_cast<int>(w - static_cast<long long>(t) * nseg);
    const int c_first = seg * 32 * CH + lane;
    const int32_t* slots = inv + static_cast<size_t>(t) * k;
    uint4* out = y + static_cast<size_t>(t) * nvec;
    if (KS > 0) {
      int r[KS > 0 ? KS : 1];
      uint4 v[KS > 0 ? KS : 1][CH], vs[CH];
#pragma unroll
      for (int sl = 0; sl < KS; ++sl) r[sl] = __ldg(slots + sl);
#pragma unroll
      for (int sl = 0; sl < KS; ++sl) {
        const uint4* row = yp + static_cast<size_t>(r[sl] >= 0 ? r[sl] : 0) * nvec;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int i = c_first + 32 * c;
          v[sl][c] = (r[sl] >= 0 && i < nvec) ? __ldg(row + i) : make_uint4(0, 0, 0, 0);
        }
      }
      if (ys != nullptr) {
        const uint4* row = ys + static_cast<size_t>(t) * nvec;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int i = c_first + 32 * c;
          vs[c] = i < nvec ? __ldg(row + i) : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int i = c_first + 32 * c;
        if (i >= nvec) continue;
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.f;
#pragma unroll
        for (int sl = 0; sl < KS; ++sl)
          if (r[sl] >= 0) add_chunk<BF16>(acc, v[sl][c]);
        if (ys != nullptr) add_chunk<BF16>(acc, vs[c]);
        out[i] = pack_chunk<BF16>(acc);
      }
    } else {
      // any k (e.g. the dense [T, E] inverse of expert choice): lanes read 32 slots at a
      // time, a ballot marks the used ones, and they are added in slot order
      const int c0 = c_first, c1 = c0 + 32;
      const bool h0 = c0 < nvec, h1 = c1 < nvec;
      float a0[8], a1[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) a0[q] = a1[q] = 0.f;
      for (int base = 0; base < k; base += 32) {
        const int mine = (base + lane < k) ? __ldg(slots + base + lane) : -1;
        unsigned used = __ballot_sync(0xffffffffu, mine >= 0);
        while (used) {
          const int j = __ffs(used) - 1;
          used &= used - 1;
          const int r = __shfl_sync(0xffffffffu, mine, j);
          const uint4* row = yp + static_cast<size_t>(r) * nvec;
          if (h0) add_chunk<BF16>(a0, __ldg(row + c0));
          if (h1) add_chunk<BF16>(a1, __ldg(row + c1));
        }
      }
      if (ys != nullptr) {
        const uint4* row = ys + static_cast<size_t>(t) * nvec;
        if (h0) add_chunk<BF16>(a0, __ldg(row + c0));
        if (h1) add_chunk<BF16>(a1, __ldg(row + c1));
      }
      if (h0) out[c0] = pack_chunk<BF16>(a0);
      if (h1) out[c1] = pack_chunk<BF16>(a1);
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
                  int row_bytes, int max_rows, void* xp, int num_sms, cudaStream_t stream,
                  DeviceError* to_f16_err) {
  if (max_rows <= 0) return MOE_OK;
  if (to_f16_err != nullptr)
    return launch_pdl(gather_rows_f16_kernel, dim3(grid_for_rows(max_rows, num_sms)),
                      dim3(kMoveThreads), 0, stream, static_cast<const uint4*>(x), perm, offsets,
                      E, k, row_bytes / 16, static_cast<uint4*>(xp), to_f16_err) == cudaSuccess
               ? MOE_OK : MOE_ERR_CUDA;
  return launch_pdl(gather_rows_kernel, dim3(grid_for_rows(max_rows, num_sms)), dim3(kMoveThreads),
                    0, stream, static_cast<const uint4*>(x), perm, offsets, E, k, row_bytes / 16,
                    static_cast<uint4*>(xp)) == cudaSuccess
             ? MOE_OK : MOE_ERR_CUDA;
}

int launch_gather_tokens(const void* x, const int32_t* inv, int T, int row_bytes, void* xp,
                         void* y, int num_sms, cudaStream_t stream) {
  if (T <= 0) return MOE_OK;
  return launch_pdl(gather_tokens_kernel, dim3(grid_for_rows(T, num_sms)), dim3(kMoveThreads), 0,
                    stream, static_cast<const uint4*>(x), inv, T, row_bytes / 16,
                    static_cast<uint4*>(xp), static_cast<uint4*>(y)) == cudaSuccess
             ? MOE_OK : MOE_ERR_CUDA;
}

template <bool BF16>
cudaError_t combine_dispatch_k(int grid, const uint4* yp, const int32_t* inv, const uint4* ys,
                               uint4* y, int T, int k, int nvec, cudaStream_t stream) {
  auto go = [&](auto kernel) {
    return launch_pdl(kernel, dim3(grid), dim3(kMoveThreads), 0, stream, yp, inv, ys, y, T, k,
                      nvec);
  };
  switch (k) {
    case 1: return go(combine_kernel<BF16, 1>);
    case 2: return go(combine_kernel<BF16, 2>);
    case 4: return go(combine_kernel<BF16, 4>);
    case 6: return go(combine_kernel<BF16, 6>);
    case 8: return go(combine_kernel<BF16, 8>);
    default: return go(combine_kernel<BF16, 0>);
  }
}

int launch_combine(int dtype, const void* yp, const int32_t* inv, const void* ys, void* y, int T,
                   int k, int d, int num_sms, cudaStream_t stream) {
  if (T <= 0) return MOE_OK;
  const int row_bytes = d * (dtype == MOE_BF16 ? 2 : 4);
  const int nvec = row_bytes / 16;
  const long long warps = static_cast<long long>(T) * ((nvec + 63) / 64);
  const int grid = grid_for_rows(warps, num_sms);
  const uint4* a = static_cast<const uint4*>(yp);
  const uint4* b = static_cast<const uint4*>(ys);
  uint4* o = static_cast<uint4*>(y);
  const cudaError_t e = dtype == MOE_BF16
                            ? combine_dispatch_k<true>(grid, a, inv, b, o, T, k, nvec, stream)
                            : combine_dispatch_k<false>(grid, a, inv, b, o, T, k, nvec, stream);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
