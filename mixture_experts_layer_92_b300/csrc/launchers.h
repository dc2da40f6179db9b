// Internal host-side launchers shared between the kernel files and the C-ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"  // include/ is on the include path

namespace moe {

struct DeviceError;

// Launches `kernel` with programmatic stream serialization: its launch and set-up overlap the
// end of the previous kernel in the stream. Only for kernels that call pdl_wait() (common.cuh)
// before reading what earlier kernels wrote.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// One thread waits on an mbarrier that nothing completes (selftest.cu): the bounded wait
// records MOE_ERR_TIMEOUT at SITE_SELFTEST_WAIT in *err and returns.
int launch_wait_timeout(DeviceError* err, cudaStream_t stream);

// Sets the text moe_last_error_detail() returns on this thread; returns `status`.
int set_error_detail(int status, const char* text);

// ---------------------------------------------------------------- tcgen05 grouped GEMM
enum TcMode : int { TC_F32OUT = 0, TC_SWIGLU = 1, TC_SCALE = 2 };

struct TcArgs {
  int groups;               // routed groups G, 1..1024
  const int32_t* offsets;   // device [G+1] row offsets, or nullptr: one group of m_single rows
  int m_single;
  int n_routed;             // output columns per routed group
  int k_routed;             // reduction length (routed)
  void* out_routed;
  long long ldo_routed;     // output row stride, elements
  int has_shared;           // 1: one extra group over rows [0, m_shared) of its own A and B
  int m_shared, n_shared, k_shared;
  void* out_shared;
  long long ldo_shared;
  const int32_t* perm;      // TC_SCALE: row r is scaled by gate[perm[r]] (gate == nullptr: 1)
  const float* gate;
  const float* row_gate;    // TC_SCALE: if set, row r is scaled by row_gate[r] instead
  const float* bias;        // TC_F32OUT: per-column bias or nullptr
  const float* scale0;      // 8-bit weights: per-row scale of B0 [groups][rows] (W1 or W2)
  const float* scale1;      //                per-row scale of B1 (W3)
  int splits;               // TC_F32OUT: split-K factor (>= 1); split s writes out + s*split_stride
  int kb_per_split;         //            k-blocks (of 64) per split
  long long split_stride;   //            elements
  void* gu_routed;          // TC_SWIGLU, optional: the pre-activations G = A.W1^T and U = A.W3^T
  void* gu_shared;          //   as bf16 [rows, 2N] (G in columns 0..N-1, U in N..2N-1); out_* may
                            //   then be nullptr (H not written)
  DeviceError* err;
  int tma_out;              // set by launch_tc_gemm: bit 0 (routed) / bit 1 (shared) outputs,
                            //   bit 2 / bit 3 the G | U outputs, leave through tensor stores
  int scatter_rows;         // TC_SCALE, top-1 layers: routed row r is written at output row
                            //   perm[r] (the token: the combine folded into the epilogue)
};

// Largest group count for which launch_tc_gemm takes mt = 2 (its tile table and store
// staging then still fit in shared memory).
constexpr int kTcMt2MaxGroups = 240;

struct TcProblem {
  TcArgs args;
  const void* a;            // routed A [a_rows, k_routed] bf16
  long long a_rows;
  const void* b0;           // routed B [b_groups, b_rows, k_routed] bf16 (TC_SWIGLU: W1)
  const void* b1;           // TC_SWIGLU: W3, same shape
  long long b_rows;
  int b_groups;
  const void* a_s;          // shared A [m_shared, k_shared]
  const void* b0_s;         // shared B [b_rows_s, k_shared]
  const void* b1_s;
  long long b_rows_s;
  long long max_tiles;      // host upper bound on the tile count (sizes the grid)
  int num_sms;
};

// mt: 128-row tiles per CTA tile (1, or 2 for TC_SWIGLU / TC_SCALE with BN = 256);
// kb: K elements per pipeline stage (64: 128-byte swizzle);
// w8: B (the routed weights) are E4M3 codes with per-row scales (args.scale0/scale1),
//     expanded to fp16 in shared memory (A is fp16 too: the gather converts it, the
//     SwiGLU epilogue writes H as fp16); mt must be 1 and there is no shared expert;
// ar: rows per CTA tile, 128 (times mt), or 32 with mt = 1 (short row tiles: correct for
//     any group size, efficient when no group has more than 32 rows).
int launch_tc_gemm(int mode, int bn, int mt, int kb, bool w8, int ar, const TcProblem& p,
                   cudaStream_t stream);
// The same GEMMs (TC_SWIGLU or TC_SCALE, bf16, BN = 256, no 8-bit weights) with 256-row
// tiles on CTA pairs (tc_pair.cu); p.max_tiles counts 256-row tiles.
int launch_tc_pair_gemm(int mode, const TcProblem& p, cudaStream_t stream);

// ---------------------------------------------------------------- block-scaled expert GEMMs
// (tc_mx.cu) A: E4M3 codes [a_rows, k] with tile-atom scales `sfa` (mx_quant.cu); B: E4M3
// codes [groups, n_rows, k] or E2M1 codes packed two per byte, scales in atoms
// [groups][n_rows / 128][k / 128][512]. k % 128 == 0, n_rows % 128 == 0 (TC_SCALE: % 256).
struct MxArgs {
  int groups;
  const int32_t* offsets;   // device [groups + 1] row offsets
  int n;                    // output columns per group (TC_SWIGLU: d_ff; TC_SCALE: d)
  int n_rows;               // rows of B per group (= n)
  int k;                    // reduction length
  const uint8_t* sfa;       // activation scale atoms
  const uint8_t* sfb0;      // weight scale atoms of B0 (W1 or W2)
  const uint8_t* sfb1;      //                     of B1 (W3)
  uint8_t* out_codes;       // TC_SWIGLU: H codes [rows, n]
  uint8_t* out_atoms;       //            H scale atoms (the same row tiles)
  void* out_rows;           // TC_SCALE: bf16 [rows, ldo]
  long long ldo;
  const int32_t* perm;      // TC_SCALE gates: gate[perm[r]], or row_gate[r]
  const float* gate;
  const float* row_gate;
  DeviceError* err;
  int tma_out;              // set by launch_mx_gemm: outputs leave through tensor stores
};
struct MxProblem {
  MxArgs args;
  const void* a;
  long long a_rows;
  const void* b0;
  const void* b1;
  long long max_tiles;
  int num_sms;
};
// mode TC_SWIGLU or TC_SCALE; ar: rows per tile (128, or 32 when no group has more than
// 32 rows); bfmt: 0 = E4M3 weights, 5 = E2M1 weights.
int launch_mx_gemm(int mode, int ar, int bfmt, const MxProblem& p, cudaStream_t stream);
// E4M3 blocks of 32 of bf16 rows x [rows, K] (mx_quant.cu): codes [rows, K], scale bytes
// [rows, K / 32] (s + 127), row-major.
int launch_mx_quant_rows(const void* x, long long rows, int K, uint8_t* codes, uint8_t* scales,
                         DeviceError* err, cudaStream_t stream);
// The gathered rows Xq[r] = E4M3 blocks of x[perm[r] / k] for r < offsets[G], with the scales
// in tile atoms of TM-row tiles.
int launch_mx_gather_quant(const void* x, const int32_t* perm, const int32_t* offsets, int G,
                           int k, int K, int TM, long long max_rows, uint8_t* codes,
                           uint8_t* atoms, DeviceError* err, int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------- tcgen05 backward GEMMs
enum BwdMode : int {
  BW_DGRAD_H = 0,  // dH = dY.W2 (B = W2 read MN-major) + SwiGLU backward and dgate partials
  BW_DGRAD_X = 1,  // dX = [dG dU].[W1; W3] (B = W1 / W3 read MN-major), bf16 out
  BW_WGRAD = 2,    // dW[g] = A_g^T . B_g over the rows of group g (both read MN-major), fp32 out
};

struct BwdArgs {
  int groups;               // row groups (expert segments), 1..1024
  const int32_t* offsets;   // device [groups+1] row offsets, or nullptr: one group of m_single
  int m_single;
  int M;                    // BW_WGRAD: output rows (A's columns)
  int N;                    // output columns
  int K;                    // DGRAD: reduction length (A's columns)
  int k_split;              // BW_DGRAD_X: k < k_split reads B0 (W1), k >= k_split reads B1 (W3)
  void* out;                // DGRAD_X: bf16 [rows, N] (ldo); WGRAD: fp32 [groups, m_split, N]
  long long ldo;
  void* out1;               // WGRAD: rows m >= m_split go to out1 [groups, M - m_split, N]
  int m_split;
  // BW_DGRAD_H epilogue
  const void* gu;           // G | U of the forward, bf16 [rows, 2N]
  void* dgu;                // out: dG | dU, bf16 [rows, 2N]
  void* h;                  // out: H = silu(G) U, bf16 [rows, N]
  float* dg_part;           // out (nullable): per row, column tile and column half,
  int n_tiles;              //   sum_f dH_raw * H: [rows, n_tiles] with n_tiles = 2 * tiles
  const int32_t* perm;      // gate of row r = gate[perm[r]], or gate[r] when perm == nullptr
                            //   (expert-choice rows); gate == nullptr: 1
  const float* gate;
  DeviceError* err;
  int tma_out;              // set by launch_bwd_gemm (DGRAD): outputs through tensor stores
};

struct BwdProblem {
  BwdArgs args;
  const void* a;            // A: DGRAD [a_rows, K] K-major; WGRAD [a_rows, a_inner] MN-major
  long long a_rows, a_inner;
  const void* b0;           // DGRAD: weights [b_groups, b_rows, b_inner]; WGRAD: [b_rows, b_inner]
  const void* b1;           // DGRAD_X: W3 (same shape as b0)
  long long b_rows, b_inner;
  int b_groups;
  long long max_tiles;
  int num_sms;
};

// mt: 128-row output tiles per CTA tile (2 only for BW_WGRAD).
int launch_bwd_gemm(int mode, int bn, int mt, const BwdProblem& p, cudaStream_t stream);

// Non-GEMM steps of the backward pass (backward.cu)
// dyp[r] = dy[perm[r] / k], dO[r] = g_r * dy[perm[r] / k] (bf16), r < offsets[E], with
// g_r = gate[perm[r]] (top-k: perm holds assignments) or gate[r] (gate_by_row: expert-choice
// rows, perm holds tokens and k = 1)
int launch_gather_dy(const void* dy, const int32_t* perm, const int32_t* offsets, const float* gate,
                     int E, int k, int gate_by_row, int d, int max_rows, void* dyp, void* dO,
                     int num_sms, cudaStream_t stream);
// dgate[a] = sum_j dg_part[inv[a]][j] (fixed order), 0 for a dropped assignment; inv == NULL:
// dgate[r] = sum_j dg_part[r][j] for every row r < A (expert-choice rows)
int launch_dgate(const float* dg_part, int n_tiles, const int32_t* inv, int A, float* dgate,
                 cudaStream_t stream);
// dl = dJ/dlogits [T, E] (fp32, and a bf16 copy) from the gate, balance and z-loss terms;
// expert choice (gate_mode MOE_GATE_EXPERT_CHOICE): idx = inv [T, E], dgate per row
int launch_dlogits(const float* logits, const int32_t* idx, const float* dgate,
                   const int32_t* counts, int T, int E, int k, int gate_mode, float alpha,
                   float beta, float d_aux, float d_z, float* dl, void* dl16, cudaStream_t stream);
// out[e] = sum over t (in order) of dl[t][e]
int launch_column_sum(const float* dl, int T, int E, float* out, cudaStream_t stream);
// dx[t] = sum_s [inv >= 0] dxp[inv[t*k+s]] + dxr[t] (+ dxs[t]), fp32 sums, bf16 out
int launch_dx_combine(const void* dxp, const int32_t* inv, const void* dxr, const void* dxs,
                      void* dx, int T, int k, int d, int num_sms, cudaStream_t stream);

// fp32 layers' backward (backward_f32.cu): one thread per output element, fixed-order sums.
// Rows of group g are offsets[g] .. offsets[g+1] (offsets == nullptr: one group of m_single).
int launch_f32_gu(const float* a, const int32_t* offsets, int G, int m_single, int rows_max,
                  const float* w1, const float* w3, int F, int d, float* gu, cudaStream_t st);
int launch_f32_dh(const float* dyp, const int32_t* offsets, int G, int m_single, int rows_max,
                  const float* w2, int F, int d, const float* gu, const int32_t* perm,
                  const float* gate, float* dgu, float* h, float* dg_part, cudaStream_t st);
int launch_f32_dx(const float* dgu, const int32_t* offsets, int G, int m_single, int rows_max,
                  const float* w1, const float* w3, int F, int d, float* dxp, cudaStream_t st);
int launch_f32_rdx(const float* dl, const float* wr, int T, int E, int d, float* dxr,
                   cudaStream_t st);
int launch_f32_wgrad(const float* a, int lda, const float* b, int ldb, const int32_t* offsets,
                     int G, int m_single, int M, int N, int m_split, float* out, float* out1,
                     cudaStream_t st);
int launch_f32_gather_dy(const float* dy, const int32_t* perm, const int32_t* offsets,
                         const float* gate, int E, int k, int gate_by_row, int d,
                         int rows_max, float* dyp, float* dO, cudaStream_t st);
int launch_f32_dx_combine(const float* dxp, const int32_t* inv, const float* dxr, const float* dxs,
                          int T, int k, int d, float* dx, cudaStream_t st);

// ---------------------------------------------------------------- CUDA-core fp32 path
struct SimtArgs {
  int groups;               // G; offsets == nullptr means one group of m_single rows
  const int32_t* offsets;
  int m_single;
  int max_rows;             // upper bound of rows in any group (grid.y)
  const float* a;           // A [*, k] fp32, rows addressed by group offsets
  const float* b0;          // B [G, n, k] (TC_SWIGLU: W1)
  const float* b1;          // TC_SWIGLU: W3
  int n, k;
  float* out;               // [*, n]
  const int32_t* perm;      // TC_SCALE gates: gate[perm[r]], or row_gate[r] if set
  const float* gate;
  const float* row_gate;
  const float* bias;        // TC_F32OUT bias
};
int launch_simt_gemm(int mode, const SimtArgs& a, cudaStream_t stream);

// ---------------------------------------------------------------- routing
int route_blocks(int T);
struct RouteArgs {
  const float* logits;      // [nsplit][T][E] fp32 partial logits, summed in split order
  int nsplit;
  size_t split_stride;      // elements between splits
  const float* bias;        // [E] added after the sum, or nullptr
  const float* select_bias; // [E] auxiliary-loss-free balancing bias (selection only), or nullptr
  float* logits_out;        // [T][E] receives the final logits, or nullptr
  float* probs_t;           // [E][T] receives the softmax probabilities, or nullptr
  int T, E, k, gate_mode;   // k = 0: no selection (probabilities and statistics only)
  int32_t* topk_idx;        // [T][k]
  float* topk_gate;         // [T][k]
  float* partials;          // [E + 1][route_blocks(T)], expert-major
  DeviceError* err;         // nullptr: no device error reporting
};
int launch_route_topk(const RouteArgs& a, cudaStream_t stream);
// The fused router (router_fused.cu): logits of bf16 x [T, d] and w_router [E, d] (E <= 256)
// on the tensor cores, split along d over the CTAs of a cluster, reduced on chip in a fixed
// order, then the routing step of launch_route_topk on them (r.logits and r.nsplit unused).
// Writes `grid` per-CTA statistic partials: r.partials [E + 1][grid].
struct RouterFusedPlan {
  int cs;       // CTAs per cluster (split of d), 1..8
  int kb_per;   // 64-wide k-blocks per CTA
  int stages;   // ring depth
  int grid;     // CTAs: ceil(T / 128) * cs
};
RouterFusedPlan router_fused_plan(int T, int d, int E);
int launch_router_fused(const RouterFusedPlan& plan, const void* x, const void* w_router,
                        const RouteArgs& r, int d, cudaStream_t stream);
int launch_update_select_bias(const int32_t* counts, float* select_bias, int T, int E, int k,
                              float gamma, cudaStream_t stream);
int launch_stats_reduce(const float* partials, int nblocks, int E, float* stats,
                        cudaStream_t stream);
// launch_stats_reduce + launch_aux_loss in one launch (T > 0); uses hdr->done_count.
int launch_stats_loss(const float* partials, int nblocks, int E, float* stats,
                      const int32_t* counts, int T, int k, float alpha, float beta, float* losses,
                      DeviceError* hdr, cudaStream_t stream);
int launch_aux_loss(const float* stats, const int32_t* counts, int T, int E, int k, float alpha,
                    float beta, float* losses, cudaStream_t stream);

// ---------------------------------------------------------------- dispatch
// blk_hist: [dispatch_max_blocks(num_sms)][E] int32 scratch; err: the workspace header
// (required: it also holds the grid-barrier words).
// loss (optional): the router's per-CTA statistics partials [E+1][nbr]; ceil((E+1)/32)
// more CTAs of the dispatch reduce them to stats[E+1] and write losses[2] from the counts
// with launch_aux_loss's arithmetic (bit-identical results), replacing launch_stats_loss.
struct DispatchLoss {
  const float* partials;
  int nbr;
  float* stats;
  int T, k;
  float alpha, beta;
  float* losses;
};
int dispatch_max_blocks(int num_sms);
int launch_dispatch(const int32_t* topk_idx, int A, int E, int C, int32_t* counts,
                    int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* dropped,
                    int32_t* blk_hist, DeviceError* err, int num_sms, cudaStream_t stream,
                    const DispatchLoss* loss = nullptr);

// ---------------------------------------------------------------- expert-choice routing
// probs_t [E][T]; writes perm/row_gate [E*C'] (C' = min(C, T)), inv [T][E] (-1 = not chosen),
// counts [E] = C', offsets [E+1], unrouted [1] = tokens no expert chose.
int launch_expert_choice(const float* probs_t, int T, int E, int C, int32_t* perm,
                         float* row_gate, int32_t* inv, int32_t* counts, int32_t* offsets,
                         int32_t* unrouted, cudaStream_t stream);

// ---------------------------------------------------------------- data movement
// to_f16_err != nullptr: x is bf16 and Xp is written as fp16 (the 8-bit-weight GEMMs'
// operand); values outside fp16's range are recorded in *to_f16_err.
int launch_gather(const void* x, const int32_t* perm, const int32_t* offsets, int E, int k,
                  int row_bytes, int max_rows, void* xp, int num_sms, cudaStream_t stream,
                  DeviceError* to_f16_err = nullptr);
int launch_combine(int dtype, const void* yp, const int32_t* inv, const void* ys, void* y, int T,
                   int k, int d, int num_sms, cudaStream_t stream);
// Top-1 layers with the combine folded into the down projection: Xp[inv[t]] = x[t] for kept
// tokens, y[t] = 0 for dropped ones (inv[t] < 0); 16-bit rows of row_bytes (multiple of 16).
int launch_gather_tokens(const void* x, const int32_t* inv, int T, int row_bytes, void* xp,
                         void* y, int num_sms, cudaStream_t stream);

}  // namespace moe
