// fp32 grouped GEMM on the CUDA cores, for fp32 layers (a tf32 tensor-core product would not
// hold fp32 accuracy). Same three epilogues as the tensor-core kernel: router logits
// (+ bias), SwiGLU silu(A.W1^T) * (A.W3^T), and the gate-scaled down projection
// ("DL S077 - Mixture of Experts (MoE) Intuition", section 1.1: w1 = gate, w3 = up,
// w2 = down; "Mixture of experts (MoE)", tirogla.com, How it works, step 4).
//
// grid = (output-column tiles, row tiles over the largest group, groups); a block whose
// rows start past its group's end exits at once. 32 x 32 output tile, K in steps of 32,
// each of the 256 threads owns a 2 x 2 patch, fp32 accumulation in a fixed K order.
#include <algorithm>

#include "common.cuh"
#include "launchers.h"

namespace moe {

namespace {

constexpr int SB = 32;  // tile edge (rows, columns and K step)

template <int MODE>
__global__ void __launch_bounds__(256) simt_gemm_kernel(const SimtArgs p) {
  __shared__ float As[SB][SB + 1];
  __shared__ float Bs[SB][SB + 1];
  __shared__ float Cs[SB][SB + 1];  // second B operand (W3) in SwiGLU mode
  const int g = blockIdx.z;
  const int lo = p.offsets ? p.offsets[g] : 0;
  const int hi = p.offsets ? p.offsets[g + 1] : p.m_single;
  const int m0 = lo + blockIdx.y * SB;
  if (m0 >= hi) return;
  const int n0 = blockIdx.x * SB;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const float* B0 = p.b0 + static_cast<size_t>(g) * p.n * p.k;
  const float* B1 = (MODE == TC_SWIGLU) ? p.b1 + static_cast<size_t>(g) * p.n * p.k : nullptr;

  float acc0[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
  float acc1[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
  for (int k0 = 0; k0 < p.k; k0 += SB) {
    for (int i = threadIdx.x; i < SB * SB; i += 256) {
      const int r = i / SB, c = i % SB;
      const int kk = k0 + c;
      const int row = m0 + r, col = n0 + r;
      As[r][c] = (row < hi && kk < p.k) ? p.a[static_cast<size_t>(row) * p.k + kk] : 0.f;
      Bs[r][c] = (col < p.n && kk < p.k) ? B0[static_cast<size_t>(col) * p.k + kk] : 0.f;
      if (MODE == TC_SWIGLU)
        Cs[r][c] = (col < p.n && kk < p.k) ? B1[static_cast<size_t>(col) * p.k + kk] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < SB; ++kk) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float a = As[ty * 2 + i][kk];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          acc0[i][j] = fmaf(a, Bs[tx * 2 + j][kk], acc0[i][j]);
          if (MODE == TC_SWIGLU) acc1[i][j] = fmaf(a, Cs[tx * 2 + j][kk], acc1[i][j]);
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int row = m0 + ty * 2 + i;
    if (row >= hi) continue;
    float scale = 1.f;
    if (MODE == TC_SCALE && p.row_gate != nullptr) scale = p.row_gate[row];
    else if (MODE == TC_SCALE && p.gate != nullptr) scale = p.gate[p.perm[row]];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int col = n0 + tx * 2 + j;
      if (col >= p.n) continue;
      float v;
      if (MODE == TC_SWIGLU) v = silu_f(acc0[i][j]) * acc1[i][j];
      else if (MODE == TC_SCALE) v = scale * acc0[i][j];
      else v = acc0[i][j] + (p.bias ? p.bias[col] : 0.f);
      p.out[static_cast<size_t>(row) * p.n + col] = v;
    }
  }
}

}  // namespace

int launch_simt_gemm(int mode, const SimtArgs& a, cudaStream_t stream) {
  if (a.max_rows <= 0 || a.n <= 0) return MOE_OK;
  dim3 grid((a.n + SB - 1) / SB, (a.max_rows + SB - 1) / SB, a.groups);
  if (grid.y > 65535u || grid.z > 65535u) return MOE_ERR_UNSUPPORTED;
  if (mode == TC_SWIGLU) simt_gemm_kernel<TC_SWIGLU><<<grid, 256, 0, stream>>>(a);
  else if (mode == TC_SCALE) simt_gemm_kernel<TC_SCALE><<<grid, 256, 0, stream>>>(a);
  else simt_gemm_kernel<TC_F32OUT><<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
