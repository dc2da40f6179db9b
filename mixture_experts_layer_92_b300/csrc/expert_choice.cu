// Expert-choice routing: every expert takes the C tokens with the highest router
// probability for it ("Mixture of Experts (MoE)", learn.starphix.com, Router Variants:
// experts choose tokens, perfect load balance). Ties go to the lower token index; inside an
// expert's segment the chosen tokens are stored in ascending token order.
//
// ec_select_kernel: one CTA (1024 threads) per expert over probs_t[e][0..T) (fp32, >= 0, so
// their bit patterns order like the values). A 4-pass radix select (8 bits per pass,
// shared-memory histogram) finds the C-th largest key K and how many of the tokens equal to
// K are needed; a final ordered pass (two block scans) keeps key > K plus the first `need`
// tokens with key == K, and writes perm / row_gate / inv. Integer decisions on the fp32
// probabilities: the result is exact for the given probabilities.
#include <algorithm>

#include "common.cuh"
#include "launchers.h"

namespace moe {

namespace {

constexpr int kEcThreads = 1024;
constexpr int kEcWarps = kEcThreads / 32;

// exclusive block scan of one int per thread; returns the thread's prefix, *total = sum
__device__ __forceinline__ int block_excl_scan(int v, int* s_w, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) s_w[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = s_w[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    s_w[lane] = w;
  }
  __syncthreads();
  const int excl = incl - v + (warp > 0 ? s_w[warp - 1] : 0);
  *total = s_w[kEcWarps - 1];
  __syncthreads();
  return excl;
}

__global__ void __launch_bounds__(kEcThreads)
ec_select_kernel(const float* __restrict__ probs_t, int T, int E, int C,
                 int32_t* __restrict__ perm, float* __restrict__ row_gate,
                 int32_t* __restrict__ inv, int32_t* __restrict__ counts,
                 int32_t* __restrict__ offsets, int keys_in_smem) {
  extern __shared__ uint32_t s_keys[];   // [T] when keys_in_smem
  __shared__ int s_hist[256];
  __shared__ int s_w[kEcWarps];
  __shared__ uint32_t s_prefix;
  __shared__ int s_need;
  const int e = blockIdx.x;
  const int tid = threadIdx.x;
  const float* col = probs_t + static_cast<size_t>(e) * T;
  const uint32_t* gkeys = reinterpret_cast<const uint32_t*>(col);
  if (keys_in_smem)
    for (int t = tid; t < T; t += kEcThreads) s_keys[t] = gkeys[t];
  const uint32_t* keys = keys_in_smem ? s_keys : gkeys;
  const int Cp = min(C, T);
  if (tid == 0) {
    counts[e] = Cp;
    offsets[e] = e * Cp;
    if (e == E - 1) offsets[E] = E * Cp;
    s_prefix = 0u;
    s_need = Cp;
  }
  __syncthreads();
  if (Cp == 0) return;

  // radix select of the Cp-th largest key, most significant byte first
  uint32_t mask = 0u;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kEcThreads) s_hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix;
    for (int t = tid; t < T; t += kEcThreads) {
      const uint32_t k = keys[t];
      if ((k & mask) == prefix) atomicAdd(&s_hist[(k >> shift) & 255u], 1);
    }
    __syncthreads();
    if (tid < 32) {
      // warp 0: lane l owns digits 255-8l .. 248-8l (descending); a suffix count over the
      // digits above finds the digit that holds the need-th largest key
      const int lane = tid;
      const int need = s_need;             // read by every lane before any lane writes it
      int cnt[8], own = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        cnt[i] = s_hist[255 - 8 * lane - i];
        own += cnt[i];
      }
      int incl = own;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      int above = incl - own;              // keys in higher digits than this lane's
      const bool mine = above < need && incl >= need;
      if (mine) {
        int dsel = 255 - 8 * lane;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (above + cnt[i] >= need) {
            dsel = 255 - 8 * lane - i;
            break;
          }
          above += cnt[i];
        }
        s_prefix = prefix | (static_cast<uint32_t>(dsel) << shift);
        s_need = need - above;
      }
    }
    mask |= 255u << shift;
    __syncthreads();
  }
  const uint32_t kth = s_prefix;   // the Cp-th largest key
  const int need_eq = s_need;      // tokens equal to kth to keep (the lowest indices)

  // ordered selection over contiguous token chunks
  const int per = (T + kEcThreads - 1) / kEcThreads;
  const int t0 = min(T, tid * per), t1 = min(T, t0 + per);
  int n_eq = 0;
  for (int t = t0; t < t1; ++t) n_eq += (keys[t] == kth);
  int total;
  const int eq_before = block_excl_scan(n_eq, s_w, &total);
  int n_sel = 0, eq_rank = eq_before;
  for (int t = t0; t < t1; ++t) {
    const uint32_t k = keys[t];
    if (k > kth) ++n_sel;
    else if (k == kth) n_sel += (eq_rank++ < need_eq);
  }
  const int sel_before = block_excl_scan(n_sel, s_w, &total);
  int pos = e * Cp + sel_before;
  eq_rank = eq_before;
  for (int t = t0; t < t1; ++t) {
    const uint32_t k = keys[t];
    bool take = k > kth;
    if (k == kth) take = (eq_rank++ < need_eq);
    if (take) {
      perm[pos] = t;
      row_gate[pos] = __uint_as_float(k);
      inv[static_cast<size_t>(t) * E + e] = pos;
      ++pos;
    }
  }
}

// tokens that no expert chose (all of inv[t][*] < 0); integer atomics: exact count
__global__ void ec_unrouted_kernel(const int32_t* __restrict__ inv, int T, int E,
                                   int32_t* __restrict__ unrouted) {
  __shared__ int s_cnt;
  if (threadIdx.x == 0) s_cnt = 0;
  __syncthreads();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < T) {
    bool any = false;
    for (int e = 0; e < E && !any; ++e) any = inv[static_cast<size_t>(t) * E + e] >= 0;
    if (!any) atomicAdd(&s_cnt, 1);
  }
  __syncthreads();
  if (threadIdx.x == 0 && s_cnt) atomicAdd(unrouted, s_cnt);
}

}  // namespace

int launch_expert_choice(const float* probs_t, int T, int E, int C, int32_t* perm,
                         float* row_gate, int32_t* inv, int32_t* counts, int32_t* offsets,
                         int32_t* unrouted, cudaStream_t stream) {
  if (cudaMemsetAsync(inv, 0xff, static_cast<size_t>(T) * E * sizeof(int32_t), stream) !=
          cudaSuccess ||
      cudaMemsetAsync(unrouted, 0, sizeof(int32_t), stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  const size_t key_bytes = static_cast<size_t>(T) * sizeof(uint32_t);
  const int in_smem = key_bytes <= 160 * 1024 ? 1 : 0;
  const size_t smem = in_smem ? key_bytes : 0;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(ec_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MOE_ERR_CUDA;
  ec_select_kernel<<<E, kEcThreads, smem, stream>>>(probs_t, T, E, C, perm, row_gate, inv, counts,
                                                    offsets, in_smem);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  if (T > 0) {
    ec_unrouted_kernel<<<(T + 255) / 256, 256, 0, stream>>>(inv, T, E, unrouted);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace moe
