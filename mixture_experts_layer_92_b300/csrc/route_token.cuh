// The per-token routing step shared by the top-k kernel (route.cu, logits read from memory)
// and the fused router (router_fused.cu, logits reduced on chip): one warp holds one
// token's final logits and computes, in this order,
//   - the softmax over all E (for the gates of softmax_all and for the balance loss's P_i),
//     written expert-major when the caller wants the probabilities (expert choice);
//   - lse = m + ln(sum) for the z-loss;
//   - the top-k selection, largest key first, the lower expert index winning ties; the key
//     is the raw logit, or the gate affinity plus a selection bias (auxiliary-loss-free
//     balancing);
//   - the gates of the selected experts in the layer's gate mode.
// "Mixture of experts (MoE)" (tirogla.com), How it works, steps 1-2 and 6; "DL S077 -
// Mixture of Experts (MoE) Intuition", section 2.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kNoIdx = 0x7fffffff;

// Order-preserving 32-bit image of a selection key: a > b as floats iff key(a) > key(b) as
// unsigned integers, -0.0 and +0.0 map to the same value, and every finite value maps above
// 0 (0 marks "not a candidate").
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = (f == 0.0f) ? 0u : __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// v[j]: the logit of expert lane + 32 j (FULL: E == 32 * JM, every slot an expert). Adds
// the token's softmax probabilities to pacc and lse^2 to lse2 (lane 0), writes
// topk_idx / topk_gate [t][0..k) (k = 0: no selection) and probs_t[e][t] if non-null.
template <int JM, bool FULL>
__device__ __forceinline__ void route_token(const float (&v)[JM], int t, int T, int E, int k,
                                            int gate_mode, const float* __restrict__ select_bias,
                                            float* __restrict__ probs_t,
                                            int32_t* __restrict__ topk_idx,
                                            float* __restrict__ topk_gate, float (&pacc)[JM],
                                            float& lse2, DeviceError* err, int err_site) {
  const int lane = threadIdx.x & 31;
  bool bad = false;
#pragma unroll
  for (int j = 0; j < JM; ++j)
    if ((FULL || lane + 32 * j < E) && !isfinite(v[j])) bad = true;
  if (__any_sync(0xffffffffu, bad)) {
    if (lane == 0) record_error(err, MOE_ERR_NONFINITE, err_site, t);
  }

  // softmax over all E, and lse for L_z
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < JM; ++j)
    if (FULL || lane + 32 * j < E) m = fmaxf(m, v[j]);
  m = warp_max(m);
  float ex[JM];
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < JM; ++j) {
    ex[j] = (FULL || lane + 32 * j < E) ? expf(v[j] - m) : 0.f;
    s += ex[j];
  }
  s = warp_sum(s);
  const float inv_s = 1.0f / s;
#pragma unroll
  for (int j = 0; j < JM; ++j) {
    const float pj = ex[j] * inv_s;
    pacc[j] += pj;
    if (probs_t != nullptr && (FULL || lane + 32 * j < E))
      probs_t[static_cast<size_t>(lane + 32 * j) * T + t] = pj;
  }
  const float lse = m + logf(s);
  if (lane == 0) lse2 += lse * lse;
  if (k == 0) return;

  // selection key: the raw logit, or the gate affinity plus the expert's selection bias --
  // sigmoid(l) for sigmoid gating, the softmax probability otherwise. The gates below never
  // include the bias.
  float key[JM];
#pragma unroll
  for (int j = 0; j < JM; ++j) {
    key[j] = v[j];
    const int e = lane + 32 * j;
    if (select_bias != nullptr && (FULL || e < E)) {
      const float a = (gate_mode == MOE_GATE_SIGMOID_TOPK) ? 1.0f / (1.0f + expf(-v[j]))
                                                           : ex[j] / s;
      key[j] = a + __ldg(select_bias + e);
    }
  }

  // k rounds of a warp arg-max over the not-yet-selected experts: each lane's best
  // candidate (a strict '>' over ascending j keeps its lowest index among equals), the
  // warp's largest key, then the lowest expert index holding it
  int slot[JM];
  uint32_t kk[JM];
#pragma unroll
  for (int j = 0; j < JM; ++j) {
    slot[j] = -1;
    kk[j] = (FULL || lane + 32 * j < E) ? order_key(key[j]) : 0u;
  }
  for (int r = 0; r < k; ++r) {
    uint32_t best = 0u;
    int bj = 0;
#pragma unroll
    for (int j = 0; j < JM; ++j)
      if (kk[j] > best) {
        best = kk[j];
        bj = j;
      }
    const uint32_t mx = __reduce_max_sync(0xffffffffu, best);
    const int bi = __reduce_min_sync(0xffffffffu, (best == mx && best != 0u) ? lane + 32 * bj
                                                                              : kNoIdx);
    if ((bi & 31) == lane) {
#pragma unroll
      for (int j = 0; j < JM; ++j)
        if (j == (bi >> 5)) {
          slot[j] = r;
          kk[j] = 0u;
        }
    }
  }

  // gates of the selected experts
  float sel_sum = 0.f;
  float aff[JM];
#pragma unroll
  for (int j = 0; j < JM; ++j) {
    aff[j] = 0.f;
    if (slot[j] >= 0) {
      if (gate_mode == MOE_GATE_SIGMOID_TOPK)
        aff[j] = 1.0f / (1.0f + expf(-v[j]));
      else
        aff[j] = ex[j];
      sel_sum += aff[j];
    }
  }
  if (gate_mode != MOE_GATE_SOFTMAX_ALL) sel_sum = warp_sum(sel_sum);
  const float inv_denom = (gate_mode == MOE_GATE_SOFTMAX_ALL) ? inv_s : 1.0f / sel_sum;
#pragma unroll
  for (int j = 0; j < JM; ++j) {
    if (slot[j] >= 0) {
      const size_t o = static_cast<size_t>(t) * k + slot[j];
      topk_idx[o] = lane + 32 * j;
      topk_gate[o] = aff[j] * inv_denom;
    }
  }
}

}  // namespace moe
