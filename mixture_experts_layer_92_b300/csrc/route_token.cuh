// The per-token routing step shared by the top-k kernel (route.cu, logits read from memory)
// and the fused router (router_fused.cu, logits reduced on chip). For every token it
// computes, in this order:
//   - the softmax over all E (for the gates of softmax_all and for the balance loss's P_i),
//     written expert-major when the caller wants the probabilities (expert choice);
//   - lse = m + ln(sum) for the z-loss;
//   - the top-k selection, largest key first, the lower expert index winning ties; the key
//     is the raw logit, or the gate affinity plus a selection bias (auxiliary-loss-free
//     balancing);
//   - the gates of the selected experts in the layer's gate mode.
// "Mixture of experts (MoE)" (tirogla.com), How it works, steps 1-2 and 6; "DL S077 -
// Mixture of Experts (MoE) Intuition", section 2.
//
// Work layout: a token is held by a group of G lanes (G = 8, 16 or 32; lane g of a group
// holds experts g, g + G, ..., g + G*(J-1)), so a warp routes 32/G tokens at once, and each
// group works on NT tokens side by side (independent dependency chains for the scheduler to
// interleave). Every reduction over a group is a butterfly of xor shuffles inside it, in a
// fixed order: results depend only on (G, J, NT) and the token-to-group assignment. The k
// winners of the selection are known to every lane of the group, and one lane stores them.
#pragma once

#include "common.cuh"

namespace moe {

template <int G>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
template <int G>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// Lanes per token group for E experts: a group's butterflies cost the same instructions
// per lane whatever its width, so narrow groups holding more values per lane route a token
// in fewer instructions (8 lanes up to E = 128, 16 up to 256, 32 beyond).
__host__ __device__ constexpr int route_group_lanes(int E) { return E <= 128 ? 8 : E <= 256 ? 16 : 32; }

// Per-lane statistics accumulated over the tokens a lane's group routes: pacc[j] sums the
// softmax probability of expert g + G*j, lse2 (lane g == 0 of a group) sums lse^2.
template <int J>
struct RouteStats {
  float pacc[J];
  float lse2;
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int j = 0; j < J; ++j) pacc[j] = 0.f;
    lse2 = 0.f;
  }
};

// One selection round over a group: the largest key among the candidates not yet taken,
// the lower expert index winning a tie (a strict '>' over ascending j inside a lane, then
// the index in the butterfly); -0.0 and +0.0 compare equal. Returns the winner's key and
// index (and, with CARRY, its `val`, e.g. the logit behind a biased key), identical in every
// lane of the group, and marks it taken in the lane that holds it.
template <int G, int J, bool CARRY>
__device__ __forceinline__ void select_round(const float (&key)[J], const float (&val)[J],
                                             const bool (&in)[J], uint32_t& taken, int g,
                                             float& wk, int& we, float& wv) {
  float b = -INFINITY, bval = 0.f;
  int be = 0x7fffffff;
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const bool c = in[j] && !((taken >> j) & 1u) && key[j] > b;
    b = c ? key[j] : b;
    be = c ? g + G * j : be;
    if (CARRY) bval = c ? val[j] : bval;
  }
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, b, o);
    const int oe = __shfl_xor_sync(0xffffffffu, be, o);
    float ov = 0.f;
    if (CARRY) ov = __shfl_xor_sync(0xffffffffu, bval, o);
    const bool take = ob > b || (ob == b && oe < be);
    b = take ? ob : b;
    be = take ? oe : be;
    if (CARRY) bval = take ? ov : bval;
  }
  if ((be & (G - 1)) == g) taken |= 1u << (be / G);
  wk = b;
  we = be;
  wv = bval;
}

template <int G, int J, int NT, bool FULL>
__device__ __forceinline__ void route_tokens(const float (&v)[NT][J], const int (&t)[NT],
                                             const bool (&valid)[NT], int T, int E, int k,
                                             int gate_mode, const float* __restrict__ select_bias,
                                             float* __restrict__ probs_t,
                                             int32_t* __restrict__ topk_idx,
                                             float* __restrict__ topk_gate, RouteStats<J>& st,
                                             DeviceError* err, int err_site) {
  const int g = threadIdx.x & (G - 1);
  // in[j]: lane slot j holds an expert
  bool in[J];
#pragma unroll
  for (int j = 0; j < J; ++j) in[j] = FULL || g + G * j < E;
  const bool raw_keys = select_bias == nullptr;
  const bool sigmoid = gate_mode == MOE_GATE_SIGMOID_TOPK;

#pragma unroll
  for (int n = 0; n < NT; ++n) {
    // 0 * v is NaN exactly when v is NaN or infinite
    float z = 0.f;
#pragma unroll
    for (int j = 0; j < J; ++j)
      if (in[j]) z = fmaf(v[n][j], 0.f, z);
    if (valid[n] && z != z) record_error(err, MOE_ERR_NONFINITE, err_site, t[n]);
  }

  // The softmax's maximum. Selecting on raw logits, the first selection round finds it (its
  // winner is the largest logit), so that round is taken here.
  float m[NT], w0k[NT], w0v[NT];
  int w0e[NT];
  uint32_t taken[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    taken[n] = 0u;
    if (raw_keys) {
      select_round<G, J, false>(v[n], v[n], in, taken[n], g, w0k[n], w0e[n], w0v[n]);
      if (k == 0) taken[n] = 0u;
      m[n] = w0k[n];
    } else {
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < J; ++j)
        if (in[j]) mx = fmaxf(mx, v[n][j]);
      m[n] = group_max<G>(mx);
    }
  }

  // softmax over all E (CUDA's fast exponential, logarithm and division: the results are
  // probabilities and gates, compared at fp32 tolerance), and lse for L_z
  float ex[NT][J], inv_s[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      ex[n][j] = in[j] ? __expf(v[n][j] - m[n]) : 0.f;
      sum += ex[n][j];
    }
    const float s = group_sum<G>(sum);
    inv_s[n] = __fdividef(1.0f, s);
    const float lse = m[n] + __logf(s);
    if (valid[n]) {
#pragma unroll
      for (int j = 0; j < J; ++j) st.pacc[j] = fmaf(ex[n][j], inv_s[n], st.pacc[j]);
      if (g == 0) st.lse2 = fmaf(lse, lse, st.lse2);
      if (probs_t != nullptr) {
#pragma unroll
        for (int j = 0; j < J; ++j)
          if (in[j]) probs_t[static_cast<size_t>(g + G * j) * T + t[n]] = ex[n][j] * inv_s[n];
      }
    }
  }
  if (k == 0) return;

#pragma unroll
  for (int n = 0; n < NT; ++n) {
    // selection keys: the raw logits, or the gate affinity plus the expert's bias (sigmoid(l)
    // for sigmoid gating, the softmax probability otherwise); gates never include the bias
    float kb[J];
#pragma unroll
    for (int j = 0; j < J; ++j) kb[j] = v[n][j];
    if (!raw_keys) {
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const float a =
            sigmoid ? __fdividef(1.0f, 1.0f + __expf(-v[n][j])) : ex[n][j] * inv_s[n];
        kb[j] = in[j] ? a + __ldg(select_bias + g + G * j) : -INFINITY;
      }
    }
    // the k rounds (rolled: this code runs a few times per block, so its size, not its
    // instruction count, sets its cost). Lane g of the group keeps round g's winner; rounds
    // from G on (k > G) are stored at once and rescaled after the sum is known.
    const size_t o0 = static_cast<size_t>(t[n]) * k;
    float sel = 0.f, myaff = 0.f;
    int mye = 0;
#pragma unroll 1
    for (int r = 0; r < k; ++r) {
      float wk, wv;
      int we;
      if (raw_keys && r == 0) {
        wv = w0k[n];
        we = w0e[n];
      } else {
        select_round<G, J, true>(kb, v[n], in, taken[n], g, wk, we, wv);
      }
      // the winner's affinity: sigmoid of its logit, or its exponential
      const float a = sigmoid ? __fdividef(1.0f, 1.0f + __expf(-wv)) : __expf(wv - m[n]);
      sel += a;
      if (r == g) {
        mye = we;
        myaff = a;
      }
      if (r >= G && valid[n] && g == 0) {
        topk_idx[o0 + r] = we;
        topk_gate[o0 + r] = a;
      }
    }
    const float denom = (gate_mode == MOE_GATE_SOFTMAX_ALL) ? inv_s[n] : __fdividef(1.0f, sel);
    if (valid[n]) {
      if (g < k) {
        topk_idx[o0 + g] = mye;
        topk_gate[o0 + g] = myaff * denom;
      }
      if (g == 0)
        for (int r = G; r < k; ++r) topk_gate[o0 + r] *= denom;
    }
  }
}

// The statistics of a warp's groups summed into every group (a fixed butterfly of xor
// shuffles across the groups); lanes 0..G-1 then hold the warp's sums.
template <int G, int J>
__device__ __forceinline__ void route_stats_warp_sum(RouteStats<J>& st) {
#pragma unroll
  for (int o = G; o < 32; o <<= 1) {
#pragma unroll
    for (int j = 0; j < J; ++j) st.pacc[j] += __shfl_xor_sync(0xffffffffu, st.pacc[j], o);
    st.lse2 += __shfl_xor_sync(0xffffffffu, st.lse2, o);
  }
}

}  // namespace moe
