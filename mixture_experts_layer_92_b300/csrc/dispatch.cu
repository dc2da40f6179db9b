// Dispatch: a stable counting sort of the T*k (token, expert) assignments by expert, with
// token order as priority and at most C assignments kept per expert.
//
// "Mixture of experts (MoE)" (tirogla.com), How it works, step 3 (group the assignments by
// expert with a counting sort, keep at most C per expert) and section Code (dispatch:
// assignments are visited in token order, which decides who is kept; the overflow is
// dropped and counted).
//
// One CTA of 1024 threads (32 warps). Warp w owns a contiguous chunk of assignments, so
// "earlier chunk" = "earlier tokens". Three phases:
//   1. per-warp histogram hist[w][e] (warp match + popcount, one writer per (w, e));
//   2. for each expert an exclusive scan over warps gives the rank of the warp's first
//      assignment to e; n_e = total; kept_e = min(n_e, C); offsets = exclusive scan of kept;
//   3. each warp re-walks its chunk in 32-wide pieces; an assignment's rank is its warp's
//      base + the running count + the number of lower lanes in the piece with the same
//      expert. rank < C -> perm[offsets[e] + rank] = a, inv[a] = that row; else inv[a] = -1.
// Integer-only and order-preserving: the outputs are bit-exact functions of the input.
#include "common.cuh"
#include "launchers.h"

namespace moe {

namespace {

constexpr int kDispThreads = 1024;
constexpr int kDispWarps = kDispThreads / 32;

__global__ void __launch_bounds__(kDispThreads)
dispatch_kernel(const int32_t* __restrict__ idx, int A, int E, int C, int32_t* __restrict__ counts,
                int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                int32_t* __restrict__ inv, int32_t* __restrict__ dropped, DeviceError* err) {
  extern __shared__ int s_mem[];
  int* hist = s_mem;                       // [kDispWarps][E]
  int* s_off = hist + kDispWarps * E;      // [E + 1]
  int* s_wsum = s_off + E + 1;             // [kDispWarps]
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;

  for (int i = tid; i < kDispWarps * E; i += kDispThreads) hist[i] = 0;
  __syncthreads();

  const int per_warp = (((A + kDispWarps - 1) / kDispWarps) + 31) & ~31;
  const int a_begin = warp * per_warp;
  const int a_end = min(A, a_begin + per_warp);

  // phase 1: histogram of this warp's chunk
  for (int base = a_begin; base < a_end; base += 32) {
    const int a = base + lane;
    int key = -1;
    if (a < a_end) {
      const int e = idx[a];
      if (e >= 0 && e < E) key = e;
      else record_error(err, MOE_ERR_INVALID, SITE_DISPATCH_INDEX, a);
    }
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    if (key >= 0 && lane == __ffs(peers) - 1) hist[warp * E + key] += __popc(peers);
  }
  __syncthreads();

  // phase 2: per-expert scan over warps, then the kept counts
  for (int e = tid; e < E; e += kDispThreads) {
    int run = 0;
    for (int w = 0; w < kDispWarps; ++w) {
      const int c = hist[w * E + e];
      hist[w * E + e] = run;
      run += c;
    }
    counts[e] = run;
    s_off[e] = min(run, C);
  }
  __syncthreads();
  // exclusive scan of s_off[0..E) (E <= 1024: one element per thread)
  {
    const int v = (tid < E) ? s_off[tid] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = s_wsum[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += n;
      }
      s_wsum[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int excl = incl - v + (warp > 0 ? s_wsum[warp - 1] : 0);
    if (tid < E) s_off[tid] = excl;
    if (tid == 0) s_off[E] = s_wsum[kDispWarps - 1];
    __syncthreads();
  }
  for (int e = tid; e <= E; e += kDispThreads) offsets[e] = s_off[e];
  if (tid == 0) *dropped = A - s_off[E];

  // phase 3: stable scatter
  for (int base = a_begin; base < a_end; base += 32) {
    const int a = base + lane;
    int key = -1;
    if (a < a_end) {
      const int e = idx[a];
      if (e >= 0 && e < E) key = e;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    if (key >= 0) {
      const int rank = hist[warp * E + key] + __popc(peers & lt_mask);
      if (rank < C) {
        const int row = s_off[key] + rank;
        perm[row] = a;
        inv[a] = row;
      } else {
        inv[a] = -1;
      }
    } else if (a < a_end) {
      inv[a] = -1;
    }
    __syncwarp();
    if (key >= 0 && lane == __ffs(peers) - 1) hist[warp * E + key] += __popc(peers);
    __syncwarp();
  }
}

}  // namespace

int launch_dispatch(const int32_t* topk_idx, int A, int E, int C, int32_t* counts,
                    int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* dropped,
                    DeviceError* err, cudaStream_t stream) {
  const size_t smem = (static_cast<size_t>(kDispWarps) * E + E + 1 + kDispWarps) * sizeof(int);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(dispatch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  dispatch_kernel<<<1, kDispThreads, smem, stream>>>(topk_idx, A, E, C, counts, offsets, perm, inv,
                                                     dropped, err);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
