// Dispatch: a stable counting sort of the T*k (token, expert) assignments by expert, with
// token order as priority and at most C assignments kept per expert.
//
// "Mixture of experts (MoE)" (tirogla.com), How it works, step 3 (group the assignments by
// expert with a counting sort, keep at most C per expert) and section Code (dispatch:
// assignments are visited in token order, which decides who is kept; the overflow is
// dropped and counted).
//
// One cooperative launch of nb CTAs x 1024 threads (all co-resident). CTA b owns the
// contiguous assignments [b*chunk, (b+1)*chunk) and warp w of it a contiguous slice, so
// "earlier CTA / earlier warp" = "earlier tokens". Phases:
//   1. per-warp histogram hist[w][e] (warp match + popcount, one writer per (w, e)); turned
//      into per-warp exclusive prefixes inside the CTA; the CTA total goes to blk_hist[b][e];
//   -- grid barrier (bounded wait) --
//   2. every CTA sums blk_hist in CTA order: base_b[e] (assignments to e in earlier CTAs) and
//      n_e; kept_e = min(n_e, C); offsets = exclusive scan of kept (CTA 0 writes them);
//   3. each warp re-walks its slice in 32-wide pieces; an assignment's rank among those
//      routed to its expert is base_b + its warp's prefix + the running count + the number
//      of lower lanes in the piece with the same expert. rank < C -> kept at offsets[e] + rank.
// Integer-only and order-preserving: the outputs are bit-exact and independent of nb.
//
// With the router's per-CTA statistics (partials [E+1][nbr]: sums of p_{t,i}, then of
// lse^2) ceil((E+1)/32) more CTAs join the grid: while the others build the histogram they
// reduce the partials to stats[E+1], one warp per row, and after the grid barrier the first
// of them forms the two losses from the counts (the balance loss alpha * E * sum_i f_i P_i
// and the z-loss beta * mean lse^2, same page, step 6). The arithmetic is route_stats.cuh's,
// which moe_aux_loss also uses: the forward's losses equal that entry point's bit for bit.
#include <algorithm>

#include "common.cuh"
#include "launchers.h"
#include "route_stats.cuh"

namespace moe {

namespace {

constexpr int kDispThreads = 1024;
constexpr int kDispWarps = kDispThreads / 32;
constexpr int kChunk = 1024;  // assignments per CTA (one 32-wide piece per warp), or a multiple

// All CTAs of the (cooperative, co-resident) grid meet here. Bounded: after kWaitLimitNs the
// waiting CTA records MOE_ERR_TIMEOUT and carries on.
__device__ __forceinline__ void grid_barrier(DeviceError* sync, unsigned nblocks) {
  __syncthreads();
  if (threadIdx.x == 0 && nblocks > 1) {
    volatile unsigned* gen = &sync->grid_gen;
    const unsigned g = *gen;
    __threadfence();
    const unsigned arrived = atomicAdd(&sync->grid_count, 1u);
    if (arrived == nblocks - 1) {
      atomicExch(&sync->grid_count, 0u);
      __threadfence();
      atomicAdd(&sync->grid_gen, 1u);
    } else {
      const unsigned long long t0 = global_timer_ns();
      while (*gen == g) {
        __nanosleep(64);
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          record_error(sync, MOE_ERR_TIMEOUT, SITE_DISPATCH_GRID_BARRIER, blockIdx.x);
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();
}

// The statistics CTAs (see the header): CTA nb_assign + c reduces rows 32c .. 32c + 31 of
// the partials (one warp per row, route_stats.cuh); after the grid barrier CTA nb_assign
// forms the losses from the counts.
__device__ void dispatch_loss_cta(const DispatchLoss& la, int E, int nb_assign,
                                  const int32_t* __restrict__ blk_hist, int* s_mem,
                                  DeviceError* err) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = static_cast<int>(blockIdx.x) - nb_assign;
  const int e = c * kDispWarps + warp;
  if (e <= E) {
    const float v = stats_row_sum_warp(la.partials + static_cast<size_t>(e) * la.nbr, la.nbr, lane);
    if (lane == 0) la.stats[e] = v;
  }
  grid_barrier(err, gridDim.x);
  if (c != 0) return;
  int* s_tot = s_mem;   // [E]: assignments per expert (the dispatch's counts)
  for (int i = threadIdx.x; i < E; i += kDispThreads) {
    int total = 0, b = 0;
    for (; b + 8 <= nb_assign; b += 8) {
      int v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldcg(blk_hist + static_cast<size_t>(b + u) * E + i);
#pragma unroll
      for (int u = 0; u < 8; ++u) total += v[u];
    }
    for (; b < nb_assign; ++b) total += __ldcg(blk_hist + static_cast<size_t>(b) * E + i);
    s_tot[i] = total;
  }
  __syncthreads();
  if (warp == 0) {
    const double sum = balance_sum_warp(s_tot, la.stats, E, lane);
    if (lane == 0)
      write_losses(sum, __ldcg(la.stats + E), la.T, E, la.k, la.alpha, la.beta, la.losses);
  }
}

__global__ void __launch_bounds__(kDispThreads)
dispatch_kernel(const int32_t* __restrict__ idx, int A, int E, int C, int chunk, int nb_assign,
                int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                int32_t* __restrict__ dropped, int32_t* __restrict__ blk_hist, DeviceError* err,
                const DispatchLoss la) {
  extern __shared__ int s_mem[];
  int* hist = s_mem;                       // [kDispWarps][E]
  int* s_base = hist + kDispWarps * E;     // [E]
  int* s_off = s_base + E;                 // [E + 1]
  int* s_wsum = s_off + E + 1;             // [kDispWarps]
  const int tid = threadIdx.x;
  pdl_launch_dependents();                 // the gather may start launching (it waits for us)
  if (static_cast<int>(blockIdx.x) >= nb_assign) {
    dispatch_loss_cta(la, E, nb_assign, blk_hist, s_mem, err);
    return;
  }
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;

  for (int i = tid; i < kDispWarps * E; i += kDispThreads) hist[i] = 0;
  __syncthreads();

  const int blk_begin = blockIdx.x * chunk;
  const int per_warp = chunk / kDispWarps;
  const int a_begin = blk_begin + warp * per_warp;
  const int a_end = min(min(A, blk_begin + chunk), a_begin + per_warp);

  // phase 1: histogram of this warp's slice
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
    __syncwarp();   // the next piece's leader may add to the same counter
  }
  __syncthreads();
  for (int e = tid; e < E; e += kDispThreads) {
    int run = 0;
    for (int w = 0; w < kDispWarps; ++w) {
      const int c = hist[w * E + e];
      hist[w * E + e] = run;
      run += c;
    }
    blk_hist[static_cast<size_t>(blockIdx.x) * E + e] = run;
  }
  grid_barrier(err, gridDim.x);

  // phase 2: this CTA's base per expert, the totals, the kept counts (eight CTAs' counts
  // loaded at a time, so their L2 latencies overlap)
  for (int e = tid; e < E; e += kDispThreads) {
    int before = 0, total = 0;
    const int nb = nb_assign, me = static_cast<int>(blockIdx.x);
    int b = 0;
    for (; b + 8 <= nb; b += 8) {
      int c[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) c[u] = __ldcg(blk_hist + static_cast<size_t>(b + u) * E + e);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (b + u < me) before += c[u];
        total += c[u];
      }
    }
    for (; b < nb; ++b) {
      const int c = __ldcg(blk_hist + static_cast<size_t>(b) * E + e);
      if (b < me) before += c;
      total += c;
    }
    s_base[e] = before;
    s_off[e] = min(total, C);
    if (blockIdx.x == 0) counts[e] = total;
  }
  __syncthreads();
  {
    // exclusive scan of s_off[0..E) (E <= 1024: one element per thread)
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
      s_wsum[lane] = w;
    }
    __syncthreads();
    const int excl = incl - v + (warp > 0 ? s_wsum[warp - 1] : 0);
    if (tid < E) s_off[tid] = excl;
    if (tid == 0) s_off[E] = s_wsum[kDispWarps - 1];
    __syncthreads();
  }
  if (blockIdx.x == 0) {
    for (int e = tid; e <= E; e += kDispThreads) offsets[e] = s_off[e];
    if (tid == 0) *dropped = A - s_off[E];
  }

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
      const int rank = s_base[key] + hist[warp * E + key] + __popc(peers & lt_mask);
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

int dispatch_max_blocks(int num_sms) { return std::max(1, std::min(num_sms, 148)); }

int launch_dispatch(const int32_t* topk_idx, int A, int E, int C, int32_t* counts,
                    int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* dropped,
                    int32_t* blk_hist, DeviceError* err, int num_sms, cudaStream_t stream,
                    const DispatchLoss* loss) {
  DispatchLoss la{};
  const int extra = (loss != nullptr && loss->partials != nullptr) ? (E + 1 + kDispWarps - 1) / kDispWarps : 0;
  if (extra) {
    la = *loss;
    if (la.nbr < 1 || la.stats == nullptr || la.losses == nullptr || la.T < 1 || la.k < 1)
      return MOE_ERR_INVALID;
  }
  const size_t smem =
      (static_cast<size_t>(kDispWarps) * E + E + E + 1 + kDispWarps) * sizeof(int);
  if (cudaFuncSetAttribute(dispatch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MOE_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_kernel, kDispThreads, smem) !=
          cudaSuccess ||
      per_sm < 1)
    return MOE_ERR_CUDA;
  // the statistics CTAs are co-resident too
  const int max_blocks = std::min(dispatch_max_blocks(num_sms), num_sms * per_sm - extra);
  if (max_blocks < 1) return MOE_ERR_CUDA;
  int chunk = kChunk;
  int nb = std::max(1, (A + chunk - 1) / chunk);
  if (nb > max_blocks) {
    chunk = ((A + max_blocks - 1) / max_blocks + kChunk - 1) / kChunk * kChunk;
    nb = std::max(1, (A + chunk - 1) / chunk);
  }
  void* args[] = {const_cast<int32_t**>(&topk_idx), &A, &E, &C, &chunk, &nb, &counts, &offsets,
                  &perm, &inv, &dropped, &blk_hist, &err, &la};
  if (cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(dispatch_kernel), dim3(nb + extra),
                                  dim3(kDispThreads), args, smem, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace moe
