/*
 * moe.h -- C ABI of libmoe: the single-GPU forward pass of one Mixture-of-Experts layer.
 *
 * The layer (pages: "Mixture of experts (MoE)", tirogla.com, section "How it works",
 * steps 1-6; "DL S077 - Mixture of Experts (MoE) Intuition", dineshblog.com, sections
 * 1.1 and 2) maps tokens x [T, d] to y [T, d]:
 *
 *   score    l_t = x_t . W_r^T (+ b)                      router weight W_r [E, d]
 *   select   top-k of l_t, descending, the lower expert index winning ties
 *   gates    softmax over all E | softmax over the k selected | sigmoid / sum over selected
 *   dispatch stable counting sort of the T*k assignments (a = t*k + slot) by expert,
 *            token order as priority, at most C kept per expert, the rest dropped
 *   compute  per-expert SwiGLU FFN  w2 (silu(w1 x) * w3 x)  as a grouped GEMM
 *   combine  y_t = sum over kept slots of g_{t,slot} * FFN_e(x_t)  (+ shared expert)
 *   balance  L_aux = alpha * E * sum_i f_i P_i,  L_z = beta * mean_t lse(l_t)^2
 *
 * Conventions for every entry point:
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise. The caller owns
 *     all buffers; the library allocates no device memory and keeps no state between
 *     calls, except a per-device cache of kernel attributes and tensor-map entry point, the
 *     fixed scratch array of moe_route_topk_noalloc, and the host pipeline handles that the
 *     caller creates and destroys (their streams and events).
 *   - Matrices are row-major and contiguous. Element type is moe_shape.dtype (fp32 or
 *     bf16) for x, weights, y and the permuted buffers; logits, gates, statistics and
 *     losses are always fp32; indices and counts are int32.
 *   - Data pointers must be 16-byte aligned, and d * sizeof(dtype) must be a multiple of
 *     16 bytes; for bf16, d, d_ff and d_ff_shared must be multiples of 8 (TMA strides).
 *   - Calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy default stream)
 *     and never synchronise the host: counts, drops and losses stay on the device.
 *   - Return value: MOE_OK, or a negative moe_status found on the host before any launch
 *     (invalid arguments, workspace too small) or reported by a launch. Errors detected on
 *     the device (an out-of-range expert index, non-finite logits, a pipeline wait that
 *     timed out) set a sticky error word in the workspace; read it with moe_get_error.
 *     The device never traps.
 *   - `ws` is a device workspace of at least moe_workspace_size(shape) bytes, 256-byte
 *     aligned. Its first 256 bytes (the error word and the dispatch kernel's grid-barrier
 *     counters) must be zero before its first use -- moe_clear_error does that; later calls
 *     keep the counters consistent by themselves. Every entry point takes the same workspace layout;
 *     calls that overlap on the GPU must not share a workspace.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID = -1,      /* bad shape, null or misaligned pointer, bad index      */
  MOE_ERR_UNSUPPORTED = -2,  /* valid but not handled (e.g. bf16 with d % 8 != 0)      */
  MOE_ERR_CUDA = -3,         /* a CUDA runtime call or launch failed                   */
  MOE_ERR_WORKSPACE = -4,    /* workspace missing, misaligned or smaller than needed   */
  MOE_ERR_TIMEOUT = -5,      /* a device pipeline wait exceeded its bound              */
  MOE_ERR_NONFINITE = -6     /* a router logit was NaN or infinite                     */
} moe_status;

/* Gate conventions ("Mixture of experts (MoE)", tirogla.com, How it works, step 1). */
typedef enum {
  MOE_GATE_SOFTMAX_ALL = 0,   /* Switch/GShard: softmax over all E, selected probs kept  */
  MOE_GATE_SOFTMAX_TOPK = 1,  /* Mixtral: softmax over the k selected logits              */
  MOE_GATE_SIGMOID_TOPK = 2,  /* DeepSeek-V3: sigmoid affinities / their sum over the k   */
  MOE_GATE_EXPERT_CHOICE = 3  /* experts choose tokens: see moe_expert_choice               */
} moe_gate_mode;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

typedef struct {
  int32_t T;            /* tokens (>= 0)                                               */
  int32_t d;            /* model width (>= 1)                                          */
  int32_t E;            /* routed experts, 1..1024                                     */
  int32_t k;            /* experts per token, 1..E                                     */
  int32_t d_ff;         /* routed expert hidden width (>= 1)                           */
  int32_t d_ff_shared;  /* always-active shared expert hidden width, 0 = none          */
  int32_t capacity;     /* C: kept assignments per expert (>= 0); C >= T means no drop */
  int32_t gate;         /* moe_gate_mode                                               */
  int32_t dtype;        /* moe_dtype of x, weights, y                                  */
  float alpha;          /* load-balancing loss coefficient                             */
  float beta;           /* router z-loss coefficient                                   */
} moe_shape;

/* Number of stages moe_forward_events records events around (see there). */
#define MOE_NUM_STAGES 8

/* C = ceil(cf * T * k / E) evaluated in double, clamped to [0, T] (C = T already means
 * no drop, since one token sends at most one assignment to an expert). ("Mixture of
 * experts (MoE)", tirogla.com, section Code: the demo's capacity; section Complexity and
 * constants: capacity factor.) Returns -1 for E < 1, k < 1, T < 0 or cf < 0. Host only. */
int moe_capacity(double cf, int32_t T, int32_t k, int32_t E);

/* Validates a shape; returns MOE_OK or the moe_status the entry points would return.
 * Host only, touches no device. */
int moe_check_shape(const moe_shape* s);

/* Workspace bytes every entry point below needs for this shape (0 if the shape is
 * invalid). Host only. */
size_t moe_workspace_size(const moe_shape* s);

/* Steps 1-2 (score, select, gates) -- "Mixture of experts (MoE)", tirogla.com, How it
 * works, steps 1-2.
 *   x [T, d], w_router [E, d] (nn.Linear layout, logits = x . w_router^T),
 *   router_bias [E] fp32 or NULL (added to the logits: it shifts selection, gates, the
 *   probabilities P_i and the z-loss).
 *   logits_in [T, E] fp32 or NULL: precomputed logits; x, w_router and router_bias are
 *   then ignored (may be NULL).
 *   logits_out [T, E] fp32 or NULL: receives the logits (fp32 accumulate).
 *   topk_idx [T, k] int32 out: selected experts per token in slot order (descending
 *   logit, ties -> lower index). topk_gate [T, k] fp32 out: gate of each slot.
 *   stats [E + 1] fp32 out or NULL: stats[i] = sum_t softmax_all(l_t)_i for i < E and
 *   stats[E] = sum_t lse(l_t)^2, each summed in a fixed order (deterministic). */
int moe_route_topk(const moe_shape* s, const void* x, const void* w_router,
                   const float* router_bias, const float* logits_in, float* logits_out,
                   int32_t* topk_idx, float* topk_gate, float* stats, void* ws,
                   size_t ws_bytes, void* stream);

/* Step 3 (dispatch) -- "Mixture of experts (MoE)", tirogla.com, How it works, step 3 and
 * section Code (dispatch): a stable counting sort of the T*k assignments by expert with
 * token order as priority; the first s->capacity of each expert are kept.
 *   topk_idx [T, k] int32, or NULL to take the top-k of logits_in [T, E] fp32 first.
 *   counts [E] out: n_e, assignments routed to e before the drop.
 *   offsets [E + 1] out: exclusive prefix sum of kept_e = min(n_e, C); R = offsets[E].
 *   perm [T * k] out: rows 0..R-1 hold the assignment id a = t*k + slot of each kept
 *   assignment, grouped by expert, increasing within an expert; rows >= R untouched.
 *   inv [T * k] out: the row of each assignment in perm, or -1 if it was dropped.
 *   dropped [1] out: sum_e max(0, n_e - C).
 * All outputs are bit-exact functions of topk_idx (no floating point). */
int moe_dispatch(const moe_shape* s, const int32_t* topk_idx, const float* logits_in,
                 int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                 int32_t* dropped, void* ws, size_t ws_bytes, void* stream);

/* Step 4 (compute) -- "Mixture of experts (MoE)", tirogla.com, How it works, step 4 and
 * Implementation notes (grouped GEMM over contiguous expert batches); "DL S077", section
 * 1.1 (SwiGLU expert: w1 = gate, w3 = up, w2 = down, no biases).
 *   x [T, d]; perm, offsets as returned by moe_dispatch.
 *   topk_gate [T, k] fp32 or NULL: row r of y_perm is scaled by topk_gate[perm[r]]
 *   (NULL: unscaled FFN outputs).
 *   w1, w3 [E, d_ff, d]; w2 [E, d, d_ff].
 *   w1s, w3s [d_ff_shared, d], w2s [d, d_ff_shared]: the shared expert, used iff
 *   s->d_ff_shared > 0 (then all three are required).
 *   y_perm [T * k, d] out: row r < R = g * FFN_e(x_t) for assignment perm[r] of expert e;
 *   rows >= R untouched.
 *   y_shared [T, d] out, required iff d_ff_shared > 0: shared expert FFN(x_t).
 * bf16 runs on the tcgen05 tensor cores with fp32 accumulation (the hidden activations are
 * rounded to bf16 between the two GEMMs); fp32 runs on the CUDA cores in fp32. */
int moe_grouped_swiglu(const moe_shape* s, const void* x, const int32_t* perm,
                       const int32_t* offsets, const float* topk_gate, const void* w1,
                       const void* w3, const void* w2, const void* w1s, const void* w3s,
                       const void* w2s, void* y_perm, void* y_shared, void* ws,
                       size_t ws_bytes, void* stream);

/* Step 5 (combine) -- "Mixture of experts (MoE)", tirogla.com, How it works, step 5:
 * y_t = sum over slots s < k with inv[t*k+s] >= 0 of y_perm[inv[t*k+s]]  (+ y_shared[t]),
 * summed in slot order in fp32, no atomics (deterministic). A fully dropped token gives
 * y_t = 0 (+ y_shared[t]). y_shared may be NULL. y [T, d] out. */
int moe_combine(const moe_shape* s, const void* y_perm, const int32_t* inv,
                const void* y_shared, void* y, void* stream);

/* Step 6 (balance) -- "Mixture of experts (MoE)", tirogla.com, How it works, step 6:
 *   losses[0] = alpha * E * sum_i f_i * P_i with f_i = counts[i] / (T * k) (pre-drop) and
 *               P_i = stats[i] / T;
 *   losses[1] = beta * stats[E] / T.
 * stats as written by moe_route_topk, counts by moe_dispatch. Accumulated in double, in a
 * fixed order. T = 0 gives losses 0. */
int moe_aux_loss(const moe_shape* s, const float* stats, const int32_t* counts,
                 float* losses, void* stream);

/* The whole layer: steps 1-6 on one stream, no host synchronisation.
 *   x [T, d], w_router [E, d], router_bias [E] or NULL, w1/w3/w2 as above,
 *   w1s/w3s/w2s or NULL (required iff d_ff_shared > 0), y [T, d] out,
 *   counts [E] / dropped [1] / losses [2] out, each may be NULL.
 * MOE_OK means every kernel was queued, not that the outputs are valid: a fault found on the
 * device (non-finite logits, an out-of-range index, a pipeline wait that ran past its 2 s
 * limit) is recorded in the workspace's sticky error word and the kernels carry on, so y,
 * counts and losses are then meaningless. Check moe_get_error(ws) after synchronising before
 * using the outputs of a call that may have failed; the word stays set until
 * moe_clear_error. */
int moe_forward(const moe_shape* s, const void* x, const void* w_router,
                const float* router_bias, const void* w1, const void* w3, const void* w2,
                const void* w1s, const void* w3s, const void* w2s, void* y,
                int32_t* counts, int32_t* dropped, float* losses, void* ws, size_t ws_bytes,
                void* stream);

/* moe_forward from and to host memory (the end-to-end call): on `stream`, copies x_host
 * [T, d] into x_dev, runs moe_forward on x_dev into y_dev, copies y_dev into y_host [T, d]
 * and, if losses_host is not NULL, the two balance losses into losses_host [2]. Returns after
 * queuing; the host buffers must stay valid (and, for asynchronous copies, be page-locked)
 * until the stream reaches the end of the call. x_dev / y_dev: device buffers of T*d
 * elements; the other arguments as in moe_forward (counts and dropped stay in the
 * workspace). Calls that overlap on the GPU need their own x_dev, y_dev and workspace.
 * Host-side argument errors return before any copy or launch. For a stream of batches whose
 * copies overlap the layer, see moe_host_pipeline below. */
int moe_forward_host(const moe_shape* s, const void* x_host, const void* w_router,
                     const float* router_bias, const void* w1, const void* w3, const void* w2,
                     const void* w1s, const void* w3s, const void* w2s, void* y_host,
                     float* losses_host, void* x_dev, void* y_dev, void* ws, size_t ws_bytes,
                     void* stream);

/* A pipeline for a stream of host batches through one layer: batch i's x is uploaded on the
 * pipeline's own upload stream, the layer runs on the caller's stream, and y (and the two
 * losses) come back on its own download stream, so the upload of batch i+1 and the download
 * of batch i-1 overlap the layer on batch i and both copy directions stay busy. It keeps two
 * slots of device buffers (x and y [T_max, d], losses [2]) in a buffer the caller provides, and
 * owns the two copy streams (non-blocking) and the events that order a slot's reuse: a slot's
 * upload waits for the layer that last read it, and its layer waits for its upload and for
 * the download that last read its outputs.
 *
 * moe_host_pipeline_buffer_size: bytes of device buffer a pipeline for shapes up to `s_max`
 * needs (0 for an invalid shape).
 * moe_host_pipeline_create: `s_max` fixes d and dtype and the largest T; `buf` is a device
 * buffer of at least moe_host_pipeline_buffer_size(s_max) bytes, 256-byte aligned, owned by
 * the caller and kept until moe_host_pipeline_destroy returns (MOE_ERR_WORKSPACE otherwise);
 * `*out` receives the handle (NULL on error). Creates its streams and events on the current
 * CUDA device, which every later call on the handle must also have current.
 * moe_host_pipeline_forward: one batch, arguments as in moe_forward_host (x_host [T, d] and
 * y_host [T, d] page-locked, losses_host [2] or NULL), with s->d and s->dtype as at create
 * and s->T <= T_max. The layer runs on `stream` with workspace `ws`; calls that share a
 * workspace must pass the same stream. Counts and dropped stay in the workspace. Returns after
 * queuing; the host buffers must stay valid until moe_host_pipeline_join's stream reaches the
 * join. Host-side argument errors return before anything is queued.
 * moe_host_pipeline_join: `stream` waits (on the device) for every download queued so far.
 * moe_host_pipeline_destroy: waits for the pipeline's queued work, then destroys its streams,
 * events and handle (the buffer stays the caller's); NULL is a no-op. */
typedef struct moe_host_pipeline moe_host_pipeline;
size_t moe_host_pipeline_buffer_size(const moe_shape* s_max);
int moe_host_pipeline_create(const moe_shape* s_max, void* buf, size_t buf_bytes,
                             moe_host_pipeline** out);
int moe_host_pipeline_forward(moe_host_pipeline* p, const moe_shape* s, const void* x_host,
                              const void* w_router, const float* router_bias, const void* w1,
                              const void* w3, const void* w2, const void* w1s, const void* w3s,
                              const void* w2s, void* y_host, float* losses_host, void* ws,
                              size_t ws_bytes, void* stream);
int moe_host_pipeline_join(moe_host_pipeline* p, void* stream);
int moe_host_pipeline_destroy(moe_host_pipeline* p);

/* moe_forward, recording events[i] (cudaEvent_t handles created by the caller) on the
 * stream before stage i and events[MOE_NUM_STAGES] after the last one, so that each
 * stage's device time can be read with cudaEventElapsedTime. Stages: 0 router GEMM,
 * 1 gates + top-k, 2 dispatch, 3 gather, 4 gate/up GEMM + SwiGLU, 5 down GEMM + gate
 * scale, 6 combine, 7 balance losses. A stage that another one absorbs runs no kernel: the
 * fused router (bf16, E <= 256) computes stage 1 in stage 0; for top-k layers the dispatch
 * also reduces the router statistics to the losses (stage 7 empty); top-1 bf16 layers
 * without a shared expert write y in the down projection's epilogue (stage 6 empty).
 * n_events must be MOE_NUM_STAGES + 1. A NULL entry
 * records nothing at that boundary, so the kernels on either side of it still overlap (each
 * kernel's launch and set-up start during the previous one's tail); an event between two
 * kernels serialises them. */
int moe_forward_events(const moe_shape* s, const void* x, const void* w_router,
                       const float* router_bias, const void* w1, const void* w3,
                       const void* w2, const void* w1s, const void* w3s, const void* w2s,
                       void* y, int32_t* counts, int32_t* dropped, float* losses, void* ws,
                       size_t ws_bytes, void* stream, void* const* events, int n_events);

/* Expert-choice routing -- "Mixture of Experts (MoE)", learn.starphix.com, Router Variants:
 * experts choose their tokens (perfect load balance). For shapes with gate =
 * MOE_GATE_EXPERT_CHOICE: the score of (t, e) is the softmax-over-all router probability;
 * expert e keeps the C' = min(capacity, T) tokens with the highest score for it (ties ->
 * lower token index), stored in ascending token order; the gate is that probability.
 *   x/w_router/router_bias or logits_in as in moe_route_topk.
 *   perm [E*C'] out: token index of each row (expert e owns rows e*C' .. (e+1)*C'-1).
 *   offsets [E+1] out: e*C'.  row_gate [E*C'] out: gate of each row.
 *   inv [T, E] out: row of (t, e), or -1 when e did not choose t.
 *   counts [E] out: C' each.  unrouted [1] out: tokens that no expert chose.
 *   stats [E+1] or NULL: as in moe_route_topk.
 * In this mode moe_forward runs router -> expert choice -> grouped SwiGLU (perm holds tokens,
 * gates per row) -> combine over inv in expert order; moe_grouped_swiglu reads perm as token
 * indices and topk_gate as the per-row gate; moe_combine reads inv as [T, E]; its
 * `dropped` output is the unrouted count; moe_route_topk and moe_dispatch refuse the mode. */
int moe_expert_choice(const moe_shape* s, const void* x, const void* w_router,
                      const float* router_bias, const float* logits_in, int32_t* perm,
                      int32_t* offsets, float* row_gate, int32_t* inv, int32_t* counts,
                      int32_t* unrouted, float* stats, void* ws, size_t ws_bytes, void* stream);

/* Auxiliary-loss-free balancing (DeepSeek-V3) -- "Mixture of experts (MoE)", tirogla.com,
 * Implementation notes: a per-expert bias is added to the scores used for top-k selection
 * only (never to the gates) and nudged after each step by load; "DL S077 - Mixture of
 * Experts (MoE) Intuition", section 8.2: up when under-used, down when over-used.
 *
 * moe_route_topk_balanced: moe_route_topk, except that expert e is ranked by
 *   affinity_e + select_bias[e], with affinity = sigmoid(l_e) for MOE_GATE_SIGMOID_TOPK and
 *   the softmax-over-all probability otherwise (ties -> lower index). Gates, statistics and
 *   logits are exactly those of moe_route_topk for the selected experts.
 *   select_bias [E] fp32 (device), read only. */
int moe_route_topk_balanced(const moe_shape* s, const void* x, const void* w_router,
                            const float* router_bias, const float* logits_in,
                            const float* select_bias, float* logits_out, int32_t* topk_idx,
                            float* topk_gate, float* stats, void* ws, size_t ws_bytes,
                            void* stream);

/* The per-step nudge: select_bias[e] += gamma if counts[e] < T*k/E, -= gamma if
 * counts[e] > T*k/E (compared exactly as counts[e]*E vs T*k), unchanged otherwise.
 * counts [E] int32: pre-drop loads as written by moe_dispatch. gamma >= 0. In place, fp32. */
int moe_update_select_bias(const moe_shape* s, const int32_t* counts, float* select_bias,
                           float gamma, void* stream);

/* moe_forward with auxiliary-loss-free balancing: routes with moe_route_topk_balanced's
 * rule on select_bias [E] (device, fp32), runs the layer, then applies
 * moe_update_select_bias with this step's counts, so the next call sees the nudged bias.
 * events/n_events as in moe_forward_events, or NULL/0 (the bias update runs in stage 7). */
int moe_forward_balanced(const moe_shape* s, const void* x, const void* w_router,
                         const float* router_bias, const void* w1, const void* w3, const void* w2,
                         const void* w1s, const void* w3s, const void* w2s, void* y,
                         int32_t* counts, int32_t* dropped, float* losses, float* select_bias,
                         float gamma, void* ws, size_t ws_bytes, void* stream,
                         void* const* events, int n_events);

/* Low-precision expert weights for weight streaming (8-bit E4M3, one fp32 scale per weight
 * row): W[e][n][k] = e4m3(wq[e][n][k]) * w_scale[e][n]. The decode-sized layers are bound by
 * the bytes of the experts they touch ("Mixture of experts (MoE)", tirogla.com, Complexity
 * and constants: all E experts' weights stay resident; "DL S077", section 4: one Mixtral
 * expert is 3 x 4096 x 14336 parameters), so halving those bytes halves their time.
 *   w1q, w3q [E, d_ff, d] and w2q [E, d, d_ff] uint8 codes; w1_scale, w3_scale [E, d_ff] and
 *   w2_scale [E, d] fp32. The tensor cores multiply fp16 copies of the weights (the E4M3 ->
 *   fp16 expansion in shared memory is exact) by fp16 activations, and the scales are applied
 *   to the fp32 accumulators. x (bf16) is converted to fp16 when it is gathered (exact for
 *   |x| in [2^-14, 65504]; smaller values round to fp16's 2^-24 grid) and H is kept in fp16.
 *   An activation or H value beyond 65504 in magnitude sets the error word to
 *   MOE_ERR_NONFINITE (the layer's output is then not valid). x and y stay bf16.
 *   Requires dtype bf16, d_ff_shared = 0, d and d_ff multiples of 16.
 * moe_grouped_swiglu_fp8w: moe_grouped_swiglu (no shared expert) on 8-bit weights.
 * moe_forward_fp8w: moe_forward on 8-bit weights (router weight stays bf16); events/n_events
 * as in moe_forward_events, or NULL/0. */
int moe_grouped_swiglu_fp8w(const moe_shape* s, const void* x, const int32_t* perm,
                            const int32_t* offsets, const float* topk_gate, const uint8_t* w1q,
                            const float* w1_scale, const uint8_t* w3q, const float* w3_scale,
                            const uint8_t* w2q, const float* w2_scale, void* y_perm, void* ws,
                            size_t ws_bytes, void* stream);
int moe_forward_fp8w(const moe_shape* s, const void* x, const void* w_router,
                     const float* router_bias, const uint8_t* w1q, const float* w1_scale,
                     const uint8_t* w3q, const float* w3_scale, const uint8_t* w2q,
                     const float* w2_scale, void* y, int32_t* counts, int32_t* dropped,
                     float* losses, void* ws, size_t ws_bytes, void* stream, void* const* events,
                     int n_events);

/* Block-scaled ("microscaling") experts -- "Mixture of Experts (MoE)", learn.starphix.com,
 * Inference Optimization, Quantization (experts stored in 8 or 4 bits, the router in 16);
 * "DL S077 - Mixture of Experts (MoE) Intuition", section 8.2 (DeepSeek-V3 in FP8). The
 * tensor cores multiply 8-bit (or 4-bit) operands whose every 32 consecutive K values share
 * one power-of-two scale 2^s, stored as the byte s + 127 (UE8M0):
 *   - weights: w1, w3 [E, d_ff, d] and w2 [E, d, d_ff] (K = the last axis) as
 *       MOE_MX_E4M3: E4M3 codes, one byte per value, [E, N, K];
 *       MOE_MX_E2M1: E2M1 codes, two per byte (the even K index in the low nibble),
 *                    [E, N, K / 2], 32-byte aligned;
 *     and their scales in 512-byte atoms [E][N / 128][K / 128][512]: the scale of weight
 *     row n, columns 32j..32j+31 is byte (n % 32) * 16 + ((n % 128) / 32) * 4 + (j % 4) of
 *     atom (e, n / 128, j / 4);
 *   - activations: the gathered x rows and the hidden rows H = silu(x W1^T) * (x W3^T) are
 *     quantized on the GPU to E4M3 blocks of 32 along K with s the smallest integer such that
 *     the block's largest magnitude is <= 448 * 2^s (clamped to [-127, 127]), codes rounded to
 *     nearest, ties to even; a non-finite x or H value sets MOE_ERR_NONFINITE in the error
 *     word.
 * The router, dispatch, combine and losses are those of moe_forward; products are exact and
 * accumulated in fp32, y is bf16. Requires dtype bf16, top-k routing, d_ff_shared = 0,
 * d % 256 == 0 and d_ff % 128 == 0 (else MOE_ERR_UNSUPPORTED).
 * moe_mx_workspace_size: workspace bytes of moe_forward_mx (0 for an invalid shape).
 * moe_forward_mx: the layer; fmt MOE_MX_E4M3 or MOE_MX_E2M1; other arguments as
 *   moe_forward_events (events/n_events may be NULL/0).
 * moe_mx_quantize: the activation quantization alone: bf16 rows x [rows, K] (K % 32 == 0) to
 *   E4M3 codes [rows, K] and scale bytes [rows, K / 32] (row-major). ws: NULL, or a
 *   workspace whose error word receives MOE_ERR_NONFINITE for a non-finite input. */
#define MOE_MX_E4M3 0
#define MOE_MX_E2M1 1
size_t moe_mx_workspace_size(const moe_shape* s);
int moe_forward_mx(const moe_shape* s, int fmt, const void* x, const void* w_router,
                   const float* router_bias, const uint8_t* w1q, const uint8_t* w1_scales,
                   const uint8_t* w3q, const uint8_t* w3_scales, const uint8_t* w2q,
                   const uint8_t* w2_scales, void* y, int32_t* counts, int32_t* dropped,
                   float* losses, void* ws, size_t ws_bytes, void* stream, void* const* events,
                   int n_events);
int moe_mx_quantize(const void* x, int64_t rows, int32_t K, uint8_t* codes, uint8_t* scales,
                    void* ws, void* stream);

/* Backward pass (training) of the layer moe_forward computes, for top-k and expert-choice
 * layers.
 * It returns the gradient of
 *     J = sum_t dy_t . y_t + d_aux * L_aux + d_z * L_z
 * with respect to every input of the layer, the routing decisions (top-k selection and
 * dispatch, i.e. which assignments are kept) held at their forward values. The load
 * fraction f_i carries no gradient and the mean router probability P_i does ("Mixture of
 * experts (MoE)", tirogla.com, How it works, step 6). The gradients follow the chain rule
 * through the forward's steps: score l = x W_r^T + b, gates (step 1's three conventions),
 * the SwiGLU experts ("DL S077", section 1.1: O = w2 (silu(w1 x) * w3 x)), the combine
 * y_t = sum g O (step 5) and the two balance losses (step 6).
 *   Inputs: the forward's inputs (x, w_router, router_bias, w1, w3, w2 and the shared
 *   expert's w1s, w3s, w2s, with the layouts of moe_forward), dy [T, d] bf16, and the loss
 *   weights d_aux, d_z (host scalars; 1 for the plain sum of the losses).
 *   Outputs (overwritten, not accumulated): dx [T, d] bf16; dw_router [E, d], dw1 and
 *   dw3 [E, d_ff, d], dw2 [E, d, d_ff] fp32; the shared expert's dw1s, dw3s [d_ff_shared, d]
 *   and dw2s [d, d_ff_shared] fp32 (required when d_ff_shared > 0, else ignored);
 *   d_router_bias [E] fp32 (nullable); dlogits [T, E] and dgate [T, k] fp32 (nullable: the
 *   intermediate gradients of the logits and of the gates, 0 for dropped assignments).
 *   An expert that receives no rows gets a zero gradient; T = 0 zeroes every gradient.
 *   Expert-choice layers (gate = MOE_GATE_EXPERT_CHOICE; "Mixture of Experts (MoE)",
 *   learn.starphix.com, Router Variants): the experts' choices (moe_expert_choice) are held
 *   fixed; row r of expert e holds token perm[r] with gate p[perm[r]][e] of the softmax over
 *   all E, so the gates' gradient reaches the logits through that softmax. dgate is then per
 *   row: [E * min(capacity, T)] in moe_expert_choice's perm order. Every expert takes the
 *   same number of tokens, so f_i is the same for all i and L_aux = alpha E f sum_i P_i =
 *   alpha E f is constant: it has no gradient (d_aux is ignored); the z-loss has its usual one.
 *   Nothing is saved between calls: the call recomputes the routing, the dispatch and the
 *   pre-activations G = Xp w1^T, U = Xp w3^T on the tensor cores, then runs the backward
 *   GEMMs (dH = dy w2 with the SwiGLU backward in its epilogue, dXp = dG w1 + dU w3, and per
 *   expert dW1 = dG^T Xp, dW3 = dU^T Xp, dW2 = (g dy)^T H; the router's dx = dl W_r and
 *   dW_r = dl^T x), reading transposed operands MN-major instead of transposing them.
 *   Precision: bf16 layers: bf16 operands, fp32 accumulation; G, U, H, dG, dU, g dy and the
 *   logit gradient (as a GEMM operand) are rounded to bf16; weight gradients are fp32. fp32
 *   layers: everything in fp32 on the CUDA cores, one thread per output element (meant for
 *   parity-scale layers), dx fp32.
 *   bf16 layers need d, d_ff and d_ff_shared
 *   multiples of 64 and E a multiple of 8 (else MOE_ERR_UNSUPPORTED); the workspace is
 *   moe_backward_workspace_size(s) bytes (a superset of the forward's; its first 256 bytes
 *   zero before first use, like the forward's).
 *   events/n_events: NULL/0, or MOE_NUM_BWD_STAGES + 1 CUDA events recorded before each
 *   stage and after the last: 0 routing + dispatch, 1 gathers of x and dy, 2 recomputed
 *   G | U, 3 dH GEMMs, 4 gate and logit gradients, 5 dX GEMMs, 6 dx combine, 7 weight
 *   gradient GEMMs.
 * Device pointers; asynchronous on `stream`; host-side argument errors return before any
 * launch, device-side errors go to the workspace error word (moe_get_error). */
#define MOE_NUM_BWD_STAGES 8
size_t moe_backward_workspace_size(const moe_shape* s);
int moe_backward(const moe_shape* s, const void* x, const void* w_router, const float* router_bias,
                 const void* w1, const void* w3, const void* w2, const void* w1s, const void* w3s,
                 const void* w2s, const void* dy, float d_aux, float d_z, void* dx,
                 float* dw_router, float* d_router_bias, float* dw1, float* dw3, float* dw2,
                 float* dw1s, float* dw3s, float* dw2s, float* dlogits, float* dgate, void* ws,
                 size_t ws_bytes, void* stream, void* const* events, int n_events);

/* moe_route_topk for precomputed logits, for callers that cannot allocate device memory.
 * (No counterpart in the pages: it is a deployment variant, not a step of the method.)
 * Some callers cannot hand the library a workspace: code running inside a host framework
 * that owns all device memory and forbids cudaMalloc (an allocation synchronises the device
 * and can stall unrelated work), or a call site with no allocator at hand. This entry point
 * computes exactly what moe_route_topk computes from logits_in -- topk_idx [T, k] int32,
 * topk_gate [T, k] fp32 and, if stats is not NULL, stats [E + 1] fp32 -- and keeps its only
 * scratch (the per-block partial sums behind stats) in a fixed 2 MiB array inside the
 * library's own device memory, so it allocates nothing.
 *   - Limit: route_blocks(T) * (E + 1) * 4 bytes must fit in 2 MiB, where route_blocks(T) =
 *     min(ceil(T / 8), 592): any T for E <= 884. Larger sizes return MOE_ERR_UNSUPPORTED
 *     with the needed and available bytes in moe_last_error_detail().
 *   - The array exists once per GPU that loads the library and is held until the process
 *     exits. Every call on a device shares it, so calls that overlap on the GPU (e.g. on two
 *     streams) race; serialise them. Each call writes the scratch before reading it.
 *   - The first call on each device looks up the array's device address (a one-time set-up
 *     with that device current); make that first call before any stream capture.
 *   - Device-side error reporting needs a workspace, so this variant does not flag
 *     non-finite logits (moe_route_topk does).
 *   - Errors found on the host, before anything is queued: MOE_ERR_INVALID for a NULL
 *     logits_in / topk_idx / topk_gate (T > 0) or any pointer not 4-byte aligned;
 *     MOE_ERR_UNSUPPORTED for expert-choice layers (they route with moe_expert_choice) and
 *     for sizes beyond the scratch.
 * Pointers are device pointers; asynchronous on `stream`. */
int moe_route_topk_noalloc(const moe_shape* s, const float* logits_in, int32_t* topk_idx,
                           float* topk_gate, float* stats, void* stream);

/* Where the forward keeps its dispatch results inside a workspace for shape `s` (host only,
 * no GPU call): byte offsets from the workspace's start of perm [T*k] (int32; rows
 * 0..offsets[E]-1 meaningful), inv [T*k] (int32) and offsets [E+1] (int32) -- what
 * moe_dispatch would return for the batch's routing, left by the last moe_forward (or
 * variant) that ran on the workspace, until the next call on it. For tests and tools that
 * inspect the routing. MOE_ERR_INVALID for an invalid shape or a NULL output pointer;
 * MOE_ERR_UNSUPPORTED for expert-choice shapes (their perm / inv differ in meaning). */
int moe_workspace_dispatch_offsets(const moe_shape* s, size_t* perm_offset, size_t* inv_offset,
                                   size_t* offsets_offset);

/* Reads (synchronising `stream`) the sticky device error word in the workspace:
 * MOE_OK, or the first moe_status a kernel recorded since the last moe_clear_error. */
int moe_get_error(const void* ws, void* stream);

/* Clears the sticky device error word (asynchronous on `stream`). */
int moe_clear_error(void* ws, void* stream);

/* Diagnostic of the failure path above (no counterpart in the pages): one device thread waits
 * on an mbarrier that nothing completes, with the bounded wait every pipeline kernel uses. The
 * wait gives up after its limit (2 s of %globaltimer), records MOE_ERR_TIMEOUT in the
 * workspace error word (moe_get_error then reports it, site 40 in moe_last_error_detail) and
 * returns; the GPU is neither trapped nor hung and the workspace is usable again after
 * moe_clear_error. `ws`: a workspace of at least 256 bytes (256-byte aligned), `ws_bytes` its
 * size. Asynchronous on `stream`; MOE_ERR_WORKSPACE for a NULL, misaligned or short workspace
 * (before any launch). */
int moe_selftest_wait_timeout(void* ws, size_t ws_bytes, void* stream);

/* Static description of a status code. */
const char* moe_status_string(int status);

/* Host-side detail of the last error returned on this thread ("" if none). */
const char* moe_last_error_detail(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
