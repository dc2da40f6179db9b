// Backward pass of fp32 layers on the CUDA cores (the bf16 path is tc_bwd.cu + backward.cu):
// the same steps and the same chain rule, one thread per output element, every sum in a fixed
// order. fp32 layers here are the parity-scale ones (a tf32 tensor-core product would not hold
// fp32 accuracy), so these kernels aim at exactness, not speed.
//
// The expert is O = w2 (silu(w1 x) * w3 x) ("DL S077 - Mixture of Experts (MoE) Intuition",
// section 1.1) over each expert's contiguous rows ("Mixture of experts (MoE)", tirogla.com, How
// it works, step 4), weighted by the gate in the combine (step 5):
//   f32_gu     G | U = Xp W1^T | Xp W3^T                       (recomputed pre-activations)
//   f32_dh     dH_raw = dYp W2; dH = g dH_raw, dG = dH U silu'(G), dU = dH silu(G); H; and the
//              per-element products dH_raw * H whose row sums are the gate gradients
//   f32_dx     dXp = dG W1 + dU W3
//   f32_rdx    dx_router = dl W_r
//   f32_wgrad  dW[g] = A_g^T B_g over the rows of group g
//   f32_gather_dy, f32_dx_combine: the row moves of the bf16 path, in fp32
#include <algorithm>

#include "common.cuh"
#include "launchers.h"

namespace moe {

namespace {

constexpr int kT = 256;

int grid_of(long long n) {
  return static_cast<int>(std::max<long long>(1, std::min<long long>((n + kT - 1) / kT, 148 * 64)));
}

// group of kept row r: the largest g with offsets[g] <= r (offsets == nullptr: one group)
__device__ __forceinline__ int group_of(const int32_t* offsets, int G, int r) {
  if (offsets == nullptr) return 0;
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (offsets[mid] <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int rows_of(const int32_t* offsets, int G, int m_single) {
  return offsets == nullptr ? m_single : offsets[G];
}

__global__ void f32_gu_kernel(const float* __restrict__ a, const int32_t* __restrict__ offsets,
                              int G, int m_single, int rows_max, const float* __restrict__ w1,
                              const float* __restrict__ w3, int F, int d, float* __restrict__ gu) {
  const int R = rows_of(offsets, G, m_single);
  const long long total = static_cast<long long>(rows_max) * F;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(i / F), f = static_cast<int>(i % F);
    if (r >= R) continue;
    const int g = group_of(offsets, G, r);
    const float* xr = a + static_cast<size_t>(r) * d;
    const float* p1 = w1 + (static_cast<size_t>(g) * F + f) * d;
    const float* p3 = w3 + (static_cast<size_t>(g) * F + f) * d;
    float sg = 0.f, su = 0.f;
    for (int j = 0; j < d; ++j) {
      sg = fmaf(xr[j], p1[j], sg);
      su = fmaf(xr[j], p3[j], su);
    }
    gu[static_cast<size_t>(r) * 2 * F + f] = sg;
    gu[static_cast<size_t>(r) * 2 * F + F + f] = su;
  }
}

__global__ void f32_dh_kernel(const float* __restrict__ dyp, const int32_t* __restrict__ offsets,
                              int G, int m_single, int rows_max, const float* __restrict__ w2,
                              int F, int d, const float* __restrict__ gu,
                              const int32_t* __restrict__ perm, const float* __restrict__ gate,
                              float* __restrict__ dgu, float* __restrict__ h,
                              float* __restrict__ dg_part) {
  const int R = rows_of(offsets, G, m_single);
  const long long total = static_cast<long long>(rows_max) * F;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(i / F), f = static_cast<int>(i % F);
    if (r >= R) continue;
    const int g = group_of(offsets, G, r);
    const float* dr = dyp + static_cast<size_t>(r) * d;
    const float* w = w2 + static_cast<size_t>(g) * d * F + f;   // W2[g][j][f], stride F
    float raw = 0.f;
    for (int j = 0; j < d; ++j) raw = fmaf(dr[j], w[static_cast<size_t>(j) * F], raw);
    const float gz = gu[static_cast<size_t>(r) * 2 * F + f];
    const float uz = gu[static_cast<size_t>(r) * 2 * F + F + f];
    const float sg = 1.0f / (1.0f + expf(-gz));
    const float si = gz * sg;
    const float dsi = sg * (1.0f + gz * (1.0f - sg));
    const float gr = gate == nullptr ? 1.0f : perm != nullptr ? gate[perm[r]] : gate[r];
    const float dh = gr * raw;
    const float hv = si * uz;
    dgu[static_cast<size_t>(r) * 2 * F + f] = dh * uz * dsi;
    dgu[static_cast<size_t>(r) * 2 * F + F + f] = dh * si;
    h[static_cast<size_t>(r) * F + f] = hv;
    if (dg_part != nullptr) dg_part[static_cast<size_t>(r) * F + f] = raw * hv;
  }
}

__global__ void f32_dx_kernel(const float* __restrict__ dgu, const int32_t* __restrict__ offsets,
                              int G, int m_single, int rows_max, const float* __restrict__ w1,
                              const float* __restrict__ w3, int F, int d, float* __restrict__ dxp) {
  const int R = rows_of(offsets, G, m_single);
  const long long total = static_cast<long long>(rows_max) * d;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(i / d), j = static_cast<int>(i % d);
    if (r >= R) continue;
    const int g = group_of(offsets, G, r);
    const float* dr = dgu + static_cast<size_t>(r) * 2 * F;
    const float* p1 = w1 + static_cast<size_t>(g) * F * d + j;   // W1[g][f][j], stride d
    const float* p3 = w3 + static_cast<size_t>(g) * F * d + j;
    float acc = 0.f;
    for (int f = 0; f < F; ++f) acc = fmaf(dr[f], p1[static_cast<size_t>(f) * d], acc);
    for (int f = 0; f < F; ++f) acc = fmaf(dr[F + f], p3[static_cast<size_t>(f) * d], acc);
    dxp[static_cast<size_t>(r) * d + j] = acc;
  }
}

__global__ void f32_rdx_kernel(const float* __restrict__ dl, const float* __restrict__ wr, int T,
                               int E, int d, float* __restrict__ dxr) {
  const long long total = static_cast<long long>(T) * d;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / d), j = static_cast<int>(i % d);
    float acc = 0.f;
    for (int e = 0; e < E; ++e)
      acc = fmaf(dl[static_cast<size_t>(t) * E + e], wr[static_cast<size_t>(e) * d + j], acc);
    dxr[i] = acc;
  }
}

// out[g][m][n] (m < m_split; rows m >= m_split go to out1[g][m - m_split][n]) =
// sum over the rows r of group g, in order, of a[r][m] * b[r][n]
__global__ void f32_wgrad_kernel(const float* __restrict__ a, int lda, const float* __restrict__ b,
                                 int ldb, const int32_t* __restrict__ offsets, int G, int m_single,
                                 int M, int N, int m_split, float* __restrict__ out,
                                 float* __restrict__ out1) {
  const long long total = static_cast<long long>(G) * M * N;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int g = static_cast<int>(i / (static_cast<long long>(M) * N));
    const long long mn = i - static_cast<long long>(g) * M * N;
    const int m = static_cast<int>(mn / N), n = static_cast<int>(mn % N);
    const int lo = offsets ? offsets[g] : 0, hi = offsets ? offsets[g + 1] : m_single;
    float acc = 0.f;
    for (int r = lo; r < hi; ++r)
      acc = fmaf(a[static_cast<size_t>(r) * lda + m], b[static_cast<size_t>(r) * ldb + n], acc);
    if (m < m_split)
      out[(static_cast<size_t>(g) * m_split + m) * N + n] = acc;
    else
      out1[(static_cast<size_t>(g) * (M - m_split) + (m - m_split)) * N + n] = acc;
  }
}

__global__ void f32_gather_dy_kernel(const float* __restrict__ dy, const int32_t* __restrict__ perm,
                                     const int32_t* __restrict__ offsets, const float* __restrict__ gate,
                                     int E, int k, int gate_by_row, int d, int rows_max,
                                     float* __restrict__ dyp, float* __restrict__ dO) {
  const int R = offsets[E];
  const long long total = static_cast<long long>(rows_max) * d;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(i / d), j = static_cast<int>(i % d);
    if (r >= R) continue;
    const int a = perm[r];
    const float v = dy[static_cast<size_t>(a / k) * d + j];
    dyp[i] = v;
    dO[i] = gate[gate_by_row ? r : a] * v;
  }
}

__global__ void f32_dx_combine_kernel(const float* __restrict__ dxp, const int32_t* __restrict__ inv,
                                      const float* __restrict__ dxr, const float* __restrict__ dxs,
                                      int T, int k, int d, float* __restrict__ dx) {
  const long long total = static_cast<long long>(T) * d;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / d), j = static_cast<int>(i % d);
    float acc = 0.f;
    for (int s = 0; s < k; ++s) {
      const int r = inv[static_cast<size_t>(t) * k + s];
      if (r >= 0) acc += dxp[static_cast<size_t>(r) * d + j];
    }
    acc += dxr[i];
    if (dxs != nullptr) acc += dxs[i];
    dx[i] = acc;
  }
}

int last_error() { return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

}  // namespace

int launch_f32_gu(const float* a, const int32_t* offsets, int G, int m_single, int rows_max,
                  const float* w1, const float* w3, int F, int d, float* gu, cudaStream_t st) {
  if (rows_max <= 0 || F <= 0) return MOE_OK;
  f32_gu_kernel<<<grid_of(static_cast<long long>(rows_max) * F), kT, 0, st>>>(
      a, offsets, G, m_single, rows_max, w1, w3, F, d, gu);
  return last_error();
}

int launch_f32_dh(const float* dyp, const int32_t* offsets, int G, int m_single, int rows_max,
                  const float* w2, int F, int d, const float* gu, const int32_t* perm,
                  const float* gate, float* dgu, float* h, float* dg_part, cudaStream_t st) {
  if (rows_max <= 0 || F <= 0) return MOE_OK;
  f32_dh_kernel<<<grid_of(static_cast<long long>(rows_max) * F), kT, 0, st>>>(
      dyp, offsets, G, m_single, rows_max, w2, F, d, gu, perm, gate, dgu, h, dg_part);
  return last_error();
}

int launch_f32_dx(const float* dgu, const int32_t* offsets, int G, int m_single, int rows_max,
                  const float* w1, const float* w3, int F, int d, float* dxp, cudaStream_t st) {
  if (rows_max <= 0) return MOE_OK;
  f32_dx_kernel<<<grid_of(static_cast<long long>(rows_max) * d), kT, 0, st>>>(
      dgu, offsets, G, m_single, rows_max, w1, w3, F, d, dxp);
  return last_error();
}

int launch_f32_rdx(const float* dl, const float* wr, int T, int E, int d, float* dxr,
                   cudaStream_t st) {
  if (T <= 0) return MOE_OK;
  f32_rdx_kernel<<<grid_of(static_cast<long long>(T) * d), kT, 0, st>>>(dl, wr, T, E, d, dxr);
  return last_error();
}

int launch_f32_wgrad(const float* a, int lda, const float* b, int ldb, const int32_t* offsets,
                     int G, int m_single, int M, int N, int m_split, float* out, float* out1,
                     cudaStream_t st) {
  f32_wgrad_kernel<<<grid_of(static_cast<long long>(G) * M * N), kT, 0, st>>>(
      a, lda, b, ldb, offsets, G, m_single, M, N, m_split, out, out1);
  return last_error();
}

int launch_f32_gather_dy(const float* dy, const int32_t* perm, const int32_t* offsets,
                         const float* gate, int E, int k, int gate_by_row, int d,
                         int rows_max, float* dyp, float* dO, cudaStream_t st) {
  if (rows_max <= 0) return MOE_OK;
  f32_gather_dy_kernel<<<grid_of(static_cast<long long>(rows_max) * d), kT, 0, st>>>(
      dy, perm, offsets, gate, E, k, gate_by_row, d, rows_max, dyp, dO);
  return last_error();
}

int launch_f32_dx_combine(const float* dxp, const int32_t* inv, const float* dxr, const float* dxs,
                          int T, int k, int d, float* dx, cudaStream_t st) {
  if (T <= 0) return MOE_OK;
  f32_dx_combine_kernel<<<grid_of(static_cast<long long>(T) * d), kT, 0, st>>>(
      dxp, inv, dxr, dxs, T, k, d, dx);
  return last_error();
}

}  // namespace moe
