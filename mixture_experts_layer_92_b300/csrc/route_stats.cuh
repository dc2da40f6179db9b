// The router statistics and the two losses ("Mixture of experts (MoE)" (tirogla.com), How
// it works, step 6: L_aux = alpha * E * sum_i f_i * P_i with f_i = n_i / (T k) and
// P_i = (1/T) sum_t p_{t,i}; the z-loss beta * (1/T) sum_t lse_t^2), shared by every kernel
// that forms them (the statistics kernels of the routing entry points, the dispatch's
// statistics CTAs, moe_aux_loss), so that all of them produce the same bits.
//
// The routing kernels leave per-CTA partial sums: partials[e][b] for e < E is the sum of
// p_{t,e} over CTA b's tokens, partials[E][b] the sum of lse_t^2. Order of the reductions:
//   stats[e] = sum over b of partials[e][b], fp32, one warp per row: lane l adds
//              b = l, l + 32, ... in order, then xor butterflies 16, 8, 4, 2, 1 (every lane
//              ends with the same bits: each butterfly step adds the same two values in
//              both lanes);
//   sum      = sum over i of n_i * stats[i], fp64 (fused multiply-add), one warp: lane l
//              takes i = l, l + 32, ..., then the butterflies.
// The fp64 part stays this short on purpose: the GPU's fp64 rate is a small fraction of its
// fp32 rate.
#pragma once

#include "common.cuh"

namespace moe {

__device__ __forceinline__ float stats_row_sum_warp(const float* __restrict__ row, int nbr,
                                                    int lane) {
  float acc = 0.f;
  int b = lane;
  // four loads in flight per lane, added in order
  for (; b + 96 < nbr; b += 128) {
    const float v0 = __ldcg(row + b), v1 = __ldcg(row + b + 32), v2 = __ldcg(row + b + 64),
                v3 = __ldcg(row + b + 96);
    acc += v0;
    acc += v1;
    acc += v2;
    acc += v3;
  }
  for (; b < nbr; b += 32) acc += __ldcg(row + b);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  return acc;
}

__device__ __forceinline__ double balance_sum_warp(const int32_t* counts, const float* stats,
                                                   int E, int lane) {
  double acc = 0.0;
  for (int i = lane; i < E; i += 32)
    acc = fma(static_cast<double>(counts[i]), static_cast<double>(__ldcg(stats + i)), acc);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  return acc;
}

// losses[0] = alpha * E * sum / (T k T), losses[1] = beta * lse2_sum / T (T = 0: both 0).
__device__ __forceinline__ void write_losses(double sum, float lse2_sum, int T, int E, int k,
                                             float alpha, float beta, float* losses) {
  if (T == 0) {
    losses[0] = 0.f;
    losses[1] = 0.f;
    return;
  }
  const double Td = static_cast<double>(T);
  losses[0] = static_cast<float>(static_cast<double>(alpha) * E * sum /
                                 (Td * static_cast<double>(k) * Td));
  losses[1] = static_cast<float>(static_cast<double>(beta) * static_cast<double>(lse2_sum) / Td);
}

}  // namespace moe
