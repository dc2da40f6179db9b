// Block-scaled ("microscaling") activations for the block-scaled expert GEMMs.
//
// "Mixture of Experts (MoE)" (learn.starphix.com), Inference Optimization, Quantization:
// experts stored in 8 or 4 bits; "DL S077 - Mixture of Experts (MoE) Intuition", section
// 8.2: DeepSeek-V3 computes in FP8. The tensor cores' block-scaled MMA multiplies 8-bit
// operands whose every 32 consecutive K values share one power-of-two scale, so the rows
// entering each expert GEMM are quantized that way:
//   s = the smallest integer with amax <= 448 * 2^s over the 32 values (clamped to
//       [-127, 127]; amax = 0 gives -127), stored as the byte s + 127;
//   code = E4M3 of v * 2^-s, rounded to nearest, ties to even (v * 2^-s is exact in fp32 for
//       bf16 inputs and never exceeds 448, so nothing saturates).
// Scale layout for the MMA ("tile atoms"): the rows of expert g are cut into tiles of TM
// rows (TM = 128, or 32 for short row tiles), numbered across experts in order (tile
// ptile[g] + m is tile m of expert g). Each (tile, 128-wide K block) owns 512 bytes; the
// scale of local row r and 32-wide K block j sits at byte (r % 32) * 16 + (r / 32) * 4 +
// (j % 4) of atom (tile * K / 128 + j / 4). The MMA copies an atom into tensor memory as
// 32 lanes x 16 bytes, replicated over the four 32-lane quarters.
#include <algorithm>

#include "common.cuh"
#include "launchers.h"

namespace moe {
namespace {

constexpr int kQThreads = 256;

// The block exponent s for the largest magnitude `amax` of 32 values, 448 = 0.875 * 2^9:
// amax = f * 2^e with f in [0.5, 1) fits 448 * 2^s iff f * 2^(e - 9 - s) <= 0.875.
__device__ __forceinline__ int mx_exponent_e4m3(float amax) {
  if (!(amax > 0.f)) return -127;
  int e;
  const float f = frexpf(amax, &e);
  const int s = e - 9 + (f > 0.875f ? 1 : 0);
  return max(-127, min(127, s));
}

// 2^-s as an fp32 value, s in [-127, 120] (every finite fp32 amax gives s <= 120).
__device__ __forceinline__ float exp2_neg(int s) { return __int_as_float((127 - s) << 23); }

// Two fp32 values -> two E4M3 codes, `lo` in the low byte (round to nearest even).
__device__ __forceinline__ uint16_t to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Quantizes the 32 fp32 values of `v` in place of 32 codes: returns the scale byte and
// writes the codes as two 16-byte vectors at `dst` (16-byte aligned).
__device__ __forceinline__ uint8_t quantize32(const float (&v)[32], uint8_t* dst, bool* nonfinite) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  if (!isfinite(amax)) *nonfinite = true;
  const int s = mx_exponent_e4m3(isfinite(amax) ? amax : 0.f);
  const float m = exp2_neg(s);
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t a = to_e4m3x2(v[4 * i] * m, v[4 * i + 1] * m);
    const uint32_t b = to_e4m3x2(v[4 * i + 2] * m, v[4 * i + 3] * m);
    w[i] = a | (b << 16);
  }
  *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  *reinterpret_cast<uint4*>(dst + 16) = make_uint4(w[4], w[5], w[6], w[7]);
  return static_cast<uint8_t>(s + 127);
}

__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16* src, float (&v)[32]) {
  const uint4* p = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 u = __ldg(p + q);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[8 * q + 2 * i] = __uint_as_float(w[i] << 16);
      v[8 * q + 2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
}

// Row-major scales: one thread per (row, 32-value block).
__global__ void __launch_bounds__(kQThreads)
mx_quant_rows_kernel(const __nv_bfloat16* __restrict__ x, long long rows, int K,
                     uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, DeviceError* err) {
  const int nb = K / 32;
  const long long i = static_cast<long long>(blockIdx.x) * kQThreads + threadIdx.x;
  if (i >= rows * nb) return;
  const long long r = i / nb;
  const int b = static_cast<int>(i - r * nb);
  float v[32];
  load_bf16x32(x + r * K + b * 32, v);
  bool bad = false;
  scales[r * nb + b] = quantize32(v, codes + r * K + b * 32, &bad);
  if (bad) record_error(err, MOE_ERR_NONFINITE, SITE_MX_NONFINITE_X, static_cast<int>(r));
}

// Gathered rows Xq[r] = quantize(x[perm[r] / k]) for r < offsets[G], scales in tile atoms.
// Every block rebuilds the tile prefix of the groups in shared memory.
__global__ void __launch_bounds__(kQThreads)
mx_gather_quant_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ perm,
                       const int32_t* __restrict__ offsets, int G, int k, int K, int TM,
                       long long max_rows, uint8_t* __restrict__ codes, uint8_t* __restrict__ atoms,
                       DeviceError* err) {
  extern __shared__ int s_q[];   // offsets [G + 1], tile prefix [G + 1]
  int* s_off = s_q;
  int* s_pt = s_q + G + 1;
  pdl_wait();
  pdl_launch_dependents();
  for (int g = threadIdx.x; g <= G; g += kQThreads) s_off[g] = offsets[g];
  __syncthreads();
  if (threadIdx.x < 32) {
    int carry = 0;
    for (int base = 0; base < G; base += 32) {
      const int g = base + threadIdx.x;
      const int tiles = g < G ? (s_off[g + 1] - s_off[g] + TM - 1) / TM : 0;
      int incl = tiles;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (static_cast<int>(threadIdx.x) >= o) incl += v;
      }
      if (g < G) s_pt[g] = carry + incl - tiles;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (threadIdx.x == 0) s_pt[G] = carry;
  }
  __syncthreads();
  const int nb = K / 32;
  const long long R = min(static_cast<long long>(s_off[G]), max_rows);
  for (long long i = static_cast<long long>(blockIdx.x) * kQThreads + threadIdx.x; i < R * nb;
       i += static_cast<long long>(gridDim.x) * kQThreads) {
    const int r = static_cast<int>(i / nb);
    const int b = static_cast<int>(i - static_cast<long long>(r) * nb);
    int lo = 0, hi = G - 1;  // the group holding row r: largest g with s_off[g] <= r
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_off[mid] <= r) lo = mid; else hi = mid - 1;
    }
    const int local = r - s_off[lo];
    const int tile = s_pt[lo] + local / TM;
    const int rr = local % TM;
    const int t = perm[r] / k;
    float v[32];
    load_bf16x32(x + static_cast<long long>(t) * K + b * 32, v);
    bool bad = false;
    const uint8_t sc = quantize32(v, codes + static_cast<long long>(r) * K + b * 32, &bad);
    atoms[(static_cast<long long>(tile) * (K / 128) + b / 4) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 +
          (b & 3)] = sc;
    if (bad) record_error(err, MOE_ERR_NONFINITE, SITE_MX_NONFINITE_X, r);
  }
}

}  // namespace

int launch_mx_quant_rows(const void* x, long long rows, int K, uint8_t* codes, uint8_t* scales,
                         DeviceError* err, cudaStream_t stream) {
  if (rows == 0) return MOE_OK;
  const long long n = rows * (K / 32);
  mx_quant_rows_kernel<<<static_cast<unsigned>((n + kQThreads - 1) / kQThreads), kQThreads, 0,
                         stream>>>(static_cast<const __nv_bfloat16*>(x), rows, K, codes, scales, err);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_mx_gather_quant(const void* x, const int32_t* perm, const int32_t* offsets, int G,
                           int k, int K, int TM, long long max_rows, uint8_t* codes,
                           uint8_t* atoms, DeviceError* err, int num_sms, cudaStream_t stream) {
  if (max_rows == 0) return MOE_OK;
  const long long n = max_rows * (K / 32);
  const long long blocks = std::min<long long>((n + kQThreads - 1) / kQThreads, 8ll * num_sms);
  const size_t smem = static_cast<size_t>(2 * (G + 1)) * sizeof(int);
  if (launch_pdl(mx_gather_quant_kernel, dim3(static_cast<unsigned>(std::max(1ll, blocks))),
                 dim3(kQThreads), smem, stream, static_cast<const __nv_bfloat16*>(x), perm,
                 offsets, G, k, K, TM, max_rows, codes, atoms, err) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace moe
