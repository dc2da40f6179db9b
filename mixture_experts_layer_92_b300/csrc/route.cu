// Gates and top-k selection (one warp per token), the router statistics needed by the
// balance losses, and the losses themselves.
//
// "Mixture of experts (MoE)" (tirogla.com), How it works:
//   step 1 (score): gate conventions -- softmax over all E (Switch, GShard), softmax over
//          only the selected logits (Mixtral), sigmoid affinities normalised over the
//          selected experts (DeepSeek-V3);
//   step 2 (select): top-k experts per token;
//   step 6 (balance): L_aux = alpha*E*sum_i f_i*P_i and the z-loss beta*mean(lse^2).
// "DL S077 - Mixture of Experts (MoE) Intuition", section 2: top-2 then softmax over the
// two selected logits.
//
// Selection compares the raw fp32 logits: largest first, the lower expert index winning a
// tie (-0.0 and +0.0 tie). Every reduction runs in a fixed order, so results are
// bit-for-bit reproducible run to run.
#include <algorithm>

#include "common.cuh"
#include "launchers.h"
#include "route_stats.cuh"
#include "route_token.cuh"

namespace moe {

namespace {

constexpr int kRouteWarps = 8;
constexpr int kRouteThreads = kRouteWarps * 32;
constexpr int kRouteMaxBlocks = 592;

// G lanes per token, J logits per lane, NT tokens per lane group at a time (route_token.cuh);
// FULL: E == G * J (no bounds predicates).
template <int G, int J, int NT, bool FULL>
__global__ void __launch_bounds__(kRouteThreads, J >= 32 ? 1 : 2)
route_topk_kernel(const float* __restrict__ logits, int nsplit, size_t split_stride,
                  const float* __restrict__ bias, const float* __restrict__ select_bias,
                  float* __restrict__ logits_out, float* __restrict__ probs_t, int T, int E,
                  int k, int gate_mode,
                  int32_t* __restrict__ topk_idx, float* __restrict__ topk_gate,
                  float* __restrict__ partials, DeviceError* err) {
  extern __shared__ float s_part[];  // [kRouteWarps][E + 1]
  constexpr int TPW = (32 / G) * NT;  // tokens per warp per iteration
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane & (G - 1);
  const int gi = lane / G;
  pdl_wait();
  pdl_launch_dependents();

  RouteStats<J> st;
  st.zero();
  const int stride = gridDim.x * kRouteWarps * TPW;
  for (int base = (blockIdx.x * kRouteWarps + warp) * TPW; base < T; base += stride) {
    float v[NT][J];
    int t[NT];
    bool valid[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      t[n] = base + gi * NT + n;
      valid[n] = t[n] < T;
      const float* row = logits + static_cast<size_t>(t[n]) * E;
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int e = g + G * j;
        v[n][j] = 0.f;
        if (valid[n] && (FULL || e < E)) {
          // split-K partial sums of the router GEMM, added in split order, then the bias
          float acc = __ldg(row + e);
          for (int sp = 1; sp < nsplit; ++sp) acc += __ldg(row + sp * split_stride + e);
          if (bias != nullptr) acc += __ldg(bias + e);
          if (logits_out != nullptr) logits_out[static_cast<size_t>(t[n]) * E + e] = acc;
          v[n][j] = acc;
        }
      }
    }
    route_tokens<G, J, NT, FULL>(v, t, valid, T, E, k, gate_mode, select_bias, probs_t, topk_idx,
                                 topk_gate, st, err, SITE_ROUTE_NONFINITE);
  }

  // per-block partial sums of p_{t,i} and lse^2: over the warp's groups, then over the warps
  // in a fixed order, stored expert-major, partials[e][block], so that the reduction below
  // reads rows
  route_stats_warp_sum<G, J>(st);
  if (lane < G) {
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int e = g + G * j;
      if (FULL || e < E) s_part[warp * (E + 1) + e] = st.pacc[j];
    }
    if (lane == 0) s_part[warp * (E + 1) + E] = st.lse2;
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    float acc = 0.f;
    for (int w = 0; w < kRouteWarps; ++w) acc += s_part[w * (E + 1) + e];
    partials[static_cast<size_t>(e) * gridDim.x + blockIdx.x] = acc;
  }
}

// stats[e] = sum over the blocks b of partials[e][b] (route_stats.cuh): one warp per row e,
// eight rows per CTA.
__global__ void __launch_bounds__(256)
stats_reduce_kernel(const float* __restrict__ partials, int nb, int E, float* __restrict__ stats) {
  const int e = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (e > E) return;   // warp-uniform
  const float v = stats_row_sum_warp(partials + static_cast<size_t>(e) * nb, nb, threadIdx.x & 31);
  if ((threadIdx.x & 31) == 0) stats[e] = v;
}

// stats as stats_reduce_kernel, and the block that finishes last (a counter in the workspace
// header) then computes the two losses from them, as aux_loss_kernel does: one launch instead
// of two. The counter goes back to 0 for the next call.
__global__ void __launch_bounds__(256)
stats_loss_kernel(const float* __restrict__ partials, int nb, int E, float* __restrict__ stats,
                  const int32_t* __restrict__ counts, int T, int k, float alpha, float beta,
                  float* __restrict__ losses, DeviceError* hdr) {
  __shared__ bool s_last;
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + (threadIdx.x >> 5);
  pdl_wait();
  pdl_launch_dependents();
  if (e <= E) {
    const float v = stats_row_sum_warp(partials + static_cast<size_t>(e) * nb, nb, lane);
    if (lane == 0) {
      stats[e] = v;
      __threadfence();
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(&hdr->done_count, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last || threadIdx.x >= 32) return;
  __threadfence();
  const double sum = balance_sum_warp(counts, stats, E, lane);
  if (lane == 0) {
    write_losses(sum, __ldcg(stats + E), T, E, k, alpha, beta, losses);
    hdr->done_count = 0u;
  }
}

// losses from stats and counts (route_stats.cuh): one warp.
__global__ void __launch_bounds__(32)
aux_loss_kernel(const float* __restrict__ stats, const int32_t* __restrict__ counts, int T, int E,
                int k, float alpha, float beta, float* __restrict__ losses) {
  const double sum = balance_sum_warp(counts, stats, E, threadIdx.x);
  if (threadIdx.x == 0) write_losses(sum, __ldcg(stats + E), T, E, k, alpha, beta, losses);
}

// Auxiliary-loss-free balancing: b_i += gamma if expert i got fewer than T*k/E assignments,
// -= gamma if more (integer comparison n_i * E vs T * k), unchanged at the mean.
__global__ void update_select_bias_kernel(const int32_t* __restrict__ counts,
                                          float* __restrict__ select_bias, int T, int E, int k,
                                          float gamma) {
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < E; e += gridDim.x * blockDim.x) {
    const long long n = static_cast<long long>(counts[e]) * E;
    const long long mean = static_cast<long long>(T) * k;
    if (n < mean) select_bias[e] = select_bias[e] + gamma;
    else if (n > mean) select_bias[e] = select_bias[e] - gamma;
  }
}

template <int G, int J, int NT, bool FULL>
int launch_full(const RouteArgs& a, cudaStream_t stream) {
  const int nb = route_blocks(a.T);
  const size_t smem = static_cast<size_t>(kRouteWarps) * (a.E + 1) * sizeof(float);
  if (launch_pdl(route_topk_kernel<G, J, NT, FULL>, dim3(nb), dim3(kRouteThreads), smem, stream,
                 a.logits, a.nsplit, a.split_stride, a.bias, a.select_bias, a.logits_out,
                 a.probs_t, a.T, a.E, a.k, a.gate_mode, a.topk_idx, a.topk_gate, a.partials,
                 a.err) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

template <int G, int J, int NT>
int launch_gj(const RouteArgs& a, cudaStream_t stream) {
  if (a.E == G * J) return launch_full<G, J, NT, true>(a, stream);
  return launch_full<G, J, NT, false>(a, stream);
}

}  // namespace

// Grid of the top-k kernel: a function of T alone, so the reduction order (and hence every
// bit of the statistics) does not depend on the device. At most 592 blocks (4 per SM on
// 148 SMs): one wave at the register count of the common E <= 128 instantiations, where 1024
// blocks took 1.4 waves (a Switch-sized batch, 16384 tokens: 15.9 us).
int route_blocks(int T) {
  const int nb = (T + kRouteWarps - 1) / kRouteWarps;
  return std::max(1, std::min(nb, kRouteMaxBlocks));
}

int launch_route_topk(const RouteArgs& a, cudaStream_t stream) {
  // lane groups as route_group_lanes(E); two tokens per group at a time while J is small
  if (a.E <= 8) return launch_gj<8, 1, 2>(a, stream);
  if (a.E <= 16) return launch_gj<8, 2, 2>(a, stream);
  if (a.E <= 32) return launch_gj<8, 4, 2>(a, stream);
  if (a.E <= 64) return launch_gj<8, 8, 1>(a, stream);
  if (a.E <= 128) return launch_gj<8, 16, 1>(a, stream);
  if (a.E <= 256) return launch_gj<16, 16, 1>(a, stream);
  const int jm = (a.E + 31) / 32;
  if (jm <= 16) return launch_gj<32, 16, 1>(a, stream);
  return launch_gj<32, 32, 1>(a, stream);
}

int launch_stats_reduce(const float* partials, int nblocks, int E, float* stats,
                        cudaStream_t stream) {
  stats_reduce_kernel<<<(E + 1 + 7) / 8, 256, 0, stream>>>(partials, nblocks, E, stats);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_update_select_bias(const int32_t* counts, float* select_bias, int T, int E, int k,
                              float gamma, cudaStream_t stream) {
  update_select_bias_kernel<<<(E + 255) / 256, 256, 0, stream>>>(counts, select_bias, T, E, k,
                                                                 gamma);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_stats_loss(const float* partials, int nblocks, int E, float* stats,
                      const int32_t* counts, int T, int k, float alpha, float beta, float* losses,
                      DeviceError* hdr, cudaStream_t stream) {
  if (launch_pdl(stats_loss_kernel, dim3((E + 1 + 7) / 8), dim3(256), 0, stream, partials, nblocks, E, stats,
                 counts, T, k, alpha, beta, losses, hdr) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

int launch_aux_loss(const float* stats, const int32_t* counts, int T, int E, int k, float alpha,
                    float beta, float* losses, cudaStream_t stream) {
  aux_loss_kernel<<<1, 32, 0, stream>>>(stats, counts, T, E, k, alpha, beta, losses);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
