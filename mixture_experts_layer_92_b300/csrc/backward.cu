// Element-wise and reduction steps of the MoE layer's backward pass (the GEMMs are in
// tc_bwd.cu). The objective is J = sum(dy * y) + d_aux * L_aux + d_z * L_z; the routing
// decisions (top-k, dispatch) carry no gradient and neither does the load fraction f_i, while
// the mean router probability P_i does ("Mixture of experts (MoE)", tirogla.com, How it works,
// step 6).
//
// gather_dy   : dyp[r] = dy[t], dO[r] = g_r dy[t] for the kept row r of assignment a = t*k+s
//               (the combine y_t = sum g O_r of step 5, differentiated with respect to O_r)
// dgate       : dJ/dg_a = dy_t . O_r = sum_f (dy_t W2)_f H_f, reduced from the per-column-tile
//               partials of the dH GEMM in a fixed order; 0 for a dropped assignment
// dlogits     : dJ/dl_t from the gates (step 1's three conventions), from L_aux through
//               P_i and from L_z through logsumexp (step 6)
// column_sum  : router-bias gradient, sum over tokens in token order
// dx_combine  : dx_t = sum over the token's kept slots of dXp[row] + the router's and the
//               shared expert's dx, fp32 sums in slot order, bf16 out
//
// Expert-choice layers ("Mixture of Experts (MoE)", learn.starphix.com, Router Variants) use
// the same kernels with rows in place of assignments: row r of expert e holds token perm[r]
// with gate p[t][e], dgate is per row, and inv is the dense [T, E] map of pairs to rows (-1:
// expert e did not choose token t), so the combine runs over E slots per token.
#include <algorithm>

#include "common.cuh"
#include "launchers.h"

namespace moe {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

int grid_for(long long warps, int num_sms) {
  const long long blocks = (warps + kWarps - 1) / kWarps;
  return static_cast<int>(std::max<long long>(1, std::min<long long>(blocks, 8ll * num_sms)));
}

__global__ void __launch_bounds__(kThreads)
gather_dy_kernel(const uint4* __restrict__ dy, const int32_t* __restrict__ perm,
                 const int32_t* __restrict__ offsets, const float* __restrict__ gate, int E,
                 int k, int gate_by_row, int nvec, uint4* __restrict__ dyp,
                 uint4* __restrict__ dO) {
  const int R = offsets[E];
  const int lane = threadIdx.x & 31;
  const int nw = gridDim.x * kWarps;
  for (int r = blockIdx.x * kWarps + (threadIdx.x >> 5); r < R; r += nw) {
    const int a = perm[r];
    const float g = gate[gate_by_row ? r : a];
    const uint4* src = dy + static_cast<size_t>(a / k) * nvec;
    uint4* d0 = dyp + static_cast<size_t>(r) * nvec;
    uint4* d1 = dO + static_cast<size_t>(r) * nvec;
    // up to U chunks per lane loaded before any is stored: a 4 KB piece of the row per round trip
    constexpr int U = 8;
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
        if (i >= nvec) continue;
        d0[i] = v[u];
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          o[q] = pack_bf16x2(g * __uint_as_float(w[q] << 16),
                             g * __uint_as_float(w[q] & 0xffff0000u));
        d1[i] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
}

__global__ void dgate_kernel(const float* __restrict__ dg_part, int n_tiles,
                             const int32_t* __restrict__ inv, int A, float* __restrict__ dgate) {
  const int a = blockIdx.x * blockDim.x + threadIdx.x;
  if (a >= A) return;
  const int r = inv != nullptr ? inv[a] : a;
  float s = 0.0f;
  if (r >= 0)
    for (int j = 0; j < n_tiles; ++j) s += dg_part[static_cast<size_t>(r) * n_tiles + j];
  dgate[a] = s;
}

// One warp per token; a per-warp shared row of E floats collects the gate term (the selected
// experts of a token are distinct, so no two slots touch the same entry).
__global__ void __launch_bounds__(kThreads)
dlogits_kernel(const float* __restrict__ logits, const int32_t* __restrict__ idx,
               const float* __restrict__ dgate, const int32_t* __restrict__ counts, int T, int E,
               int k, int gate_mode, float aux_coef, float z_coef, float* __restrict__ dl,
               __nv_bfloat16* __restrict__ dl16) {
  extern __shared__ float s_gate[];  // [kWarps][E]
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  float* gterm = s_gate + static_cast<size_t>(wid) * E;
  const int nw = gridDim.x * kWarps;
  for (int t = blockIdx.x * kWarps + wid; t < T; t += nw) {
    const float* l = logits + static_cast<size_t>(t) * E;
    const int32_t* ix = idx + static_cast<size_t>(t) * k;
    const float* dg = dgate + static_cast<size_t>(t) * k;
    float m = -INFINITY;
    for (int j = lane; j < E; j += 32) m = fmaxf(m, l[j]);
    m = warp_max(m);
    float s = 0.0f;
    for (int j = lane; j < E; j += 32) s += __expf(l[j] - m);
    s = warp_sum(s);
    const float inv_s = 1.0f / s;
    const float lse = m + __logf(s);
    // balance term: a_j = aux_coef * n_j, minus its p-weighted mean
    float pa = 0.0f;
    for (int j = lane; j < E; j += 32)
      pa += __expf(l[j] - m) * inv_s * aux_coef * static_cast<float>(counts[j]);
    pa = warp_sum(pa);
    for (int j = lane; j < E; j += 32) gterm[j] = 0.0f;
    __syncwarp();
    if (gate_mode == MOE_GATE_EXPERT_CHOICE) {
      // expert choice: idx holds inv [T, E] (row of the pair (t, j) or -1) and dgate is per
      // row; every chosen pair's gate is p_j of the softmax over all E, so as for softmax_all
      // dl_j = p_j (a_j - sum_i p_i a_i) with a_j = dgate of the pair's row, or 0
      const int32_t* iv = idx + static_cast<size_t>(t) * E;
      float c = 0.0f;
      for (int j = lane; j < E; j += 32) {
        const int r = iv[j];
        const float pa_j = r >= 0 ? __expf(l[j] - m) * inv_s * dgate[r] : 0.0f;
        gterm[j] = pa_j;
        c += pa_j;
      }
      c = warp_sum(c);
      for (int j = lane; j < E; j += 32) gterm[j] -= __expf(l[j] - m) * inv_s * c;
      __syncwarp();
    } else if (gate_mode == MOE_GATE_SOFTMAX_ALL) {
      // g_s = p_{i_s}: dl_j = p_j (a_j - sum_i p_i a_i), a = dgate scattered onto the experts
      float c = 0.0f;
      for (int sl = lane; sl < k; sl += 32) c += __expf(l[ix[sl]] - m) * inv_s * dg[sl];
      c = warp_sum(c);
      for (int j = lane; j < E; j += 32) gterm[j] = -__expf(l[j] - m) * inv_s * c;
      __syncwarp();
      for (int sl = lane; sl < k; sl += 32) {
        const int j = ix[sl];
        gterm[j] += __expf(l[j] - m) * inv_s * dg[sl];
      }
      __syncwarp();
    } else {
      // renormalised over the selected experts: softmax (top-k) or sigmoid affinities
      float msel = -INFINITY;
      if (gate_mode == MOE_GATE_SOFTMAX_TOPK) {
        for (int sl = lane; sl < k; sl += 32) msel = fmaxf(msel, l[ix[sl]]);
        msel = warp_max(msel);
      }
      float S = 0.0f;
      for (int sl = lane; sl < k; sl += 32) {
        const float z = l[ix[sl]];
        S += gate_mode == MOE_GATE_SOFTMAX_TOPK ? __expf(z - msel) : 1.0f / (1.0f + __expf(-z));
      }
      S = warp_sum(S);
      float c = 0.0f;
      for (int sl = lane; sl < k; sl += 32) {
        const float z = l[ix[sl]];
        const float a = gate_mode == MOE_GATE_SOFTMAX_TOPK ? __expf(z - msel) : 1.0f / (1.0f + __expf(-z));
        c += a / S * dg[sl];
      }
      c = warp_sum(c);
      for (int sl = lane; sl < k; sl += 32) {
        const float z = l[ix[sl]];
        float v;
        if (gate_mode == MOE_GATE_SOFTMAX_TOPK) {
          v = __expf(z - msel) / S * (dg[sl] - c);
        } else {
          const float sg = 1.0f / (1.0f + __expf(-z));
          v = (dg[sl] - c) / S * sg * (1.0f - sg);
        }
        gterm[ix[sl]] = v;
      }
      __syncwarp();
    }
    for (int j = lane; j < E; j += 32) {
      const float p = __expf(l[j] - m) * inv_s;
      const float v = gterm[j] + p * (aux_coef * static_cast<float>(counts[j]) - pa) + z_coef * lse * p;
      dl[static_cast<size_t>(t) * E + j] = v;
      dl16[static_cast<size_t>(t) * E + j] = __float2bfloat16_rn(v);
    }
    __syncwarp();
  }
}

__global__ void column_sum_kernel(const float* __restrict__ x, int T, int E, float* __restrict__ out) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  double s = 0.0;
  for (int t = 0; t < T; ++t) s += static_cast<double>(x[static_cast<size_t>(t) * E + e]);
  out[e] = static_cast<float>(s);
}

__device__ __forceinline__ void add8(float (&acc)[8], const uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    acc[2 * q] += __uint_as_float(w[q] << 16);
    acc[2 * q + 1] += __uint_as_float(w[q] & 0xffff0000u);
  }
}

__global__ void __launch_bounds__(kThreads)
dx_combine_kernel(const uint4* __restrict__ dxp, const int32_t* __restrict__ inv,
                  const uint4* __restrict__ dxr, const uint4* __restrict__ dxs,
                  uint4* __restrict__ dx, int T, int k, int nvec) {
  const int lane = threadIdx.x & 31;
  const int nseg = (nvec + 31) / 32;
  const long long total = static_cast<long long>(T) * nseg;
  const long long nw = static_cast<long long>(gridDim.x) * kWarps;
  for (long long w = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5); w < total;
       w += nw) {
    const int t = static_cast<int>(w / nseg);
    const int c = static_cast<int>(w - static_cast<long long>(t) * nseg) * 32 + lane;
    if (c >= nvec) continue;
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
    for (int s = 0; s < k; ++s) {
      const int r = __ldg(inv + static_cast<size_t>(t) * k + s);
      if (r >= 0) add8(acc, __ldg(dxp + static_cast<size_t>(r) * nvec + c));
    }
    add8(acc, __ldg(dxr + static_cast<size_t>(t) * nvec + c));
    if (dxs != nullptr) add8(acc, __ldg(dxs + static_cast<size_t>(t) * nvec + c));
    dx[static_cast<size_t>(t) * nvec + c] =
        make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                   pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
  }
}

}  // namespace

int launch_gather_dy(const void* dy, const int32_t* perm, const int32_t* offsets, const float* gate,
                     int E, int k, int gate_by_row, int d, int max_rows, void* dyp, void* dO,
                     int num_sms, cudaStream_t stream) {
  if (max_rows <= 0) return MOE_OK;
  gather_dy_kernel<<<grid_for(max_rows, num_sms), kThreads, 0, stream>>>(
      static_cast<const uint4*>(dy), perm, offsets, gate, E, k, gate_by_row, d / 8,
      static_cast<uint4*>(dyp),
      static_cast<uint4*>(dO));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_dgate(const float* dg_part, int n_tiles, const int32_t* inv, int A, float* dgate,
                 cudaStream_t stream) {
  if (A <= 0) return MOE_OK;
  dgate_kernel<<<(A + 255) / 256, 256, 0, stream>>>(dg_part, n_tiles, inv, A, dgate);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_dlogits(const float* logits, const int32_t* idx, const float* dgate,
                   const int32_t* counts, int T, int E, int k, int gate_mode, float alpha,
                   float beta, float d_aux, float d_z, float* dl, void* dl16,
                   cudaStream_t stream) {
  if (T <= 0) return MOE_OK;
  // a_j = d_aux * alpha * E * f_j / T with f_j = n_j / (T k); z: d_z * 2 beta lse / T
  const double Td = static_cast<double>(T);
  const float aux_coef = static_cast<float>(static_cast<double>(d_aux) * alpha * E / (Td * k) / Td);
  const float z_coef = static_cast<float>(static_cast<double>(d_z) * 2.0 * beta / Td);
  const size_t smem = static_cast<size_t>(kWarps) * E * sizeof(float);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(dlogits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MOE_ERR_CUDA;
  const int blocks = std::max(1, std::min((T + kWarps - 1) / kWarps, 148 * 8));
  dlogits_kernel<<<blocks, kThreads, smem, stream>>>(logits, idx, dgate, counts, T, E, k, gate_mode,
                                                     aux_coef, z_coef, dl,
                                                     static_cast<__nv_bfloat16*>(dl16));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_column_sum(const float* x, int T, int E, float* out, cudaStream_t stream) {
  column_sum_kernel<<<(E + 127) / 128, 128, 0, stream>>>(x, T, E, out);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_dx_combine(const void* dxp, const int32_t* inv, const void* dxr, const void* dxs,
                      void* dx, int T, int k, int d, int num_sms, cudaStream_t stream) {
  if (T <= 0) return MOE_OK;
  const int nvec = d / 8;
  const long long warps = static_cast<long long>(T) * ((nvec + 31) / 32);
  dx_combine_kernel<<<grid_for(warps, num_sms), kThreads, 0, stream>>>(
      static_cast<const uint4*>(dxp), inv, static_cast<const uint4*>(dxr),
      static_cast<const uint4*>(dxs), static_cast<uint4*>(dx), T, k, nvec);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
