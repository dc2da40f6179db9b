// C ABI of libmoe (declared in include/moe.h): argument checks on the host, the workspace
// layout, and the launch sequence of the forward pass on the caller's stream.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "common.cuh"
#include "launchers.h"

namespace moe {
namespace {

thread_local std::string g_detail;

int fail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_detail = buf;
  return status;
}

int ok() {
  g_detail.clear();
  return MOE_OK;
}

size_t esize(const moe_shape* s) { return s->dtype == MOE_BF16 ? 2 : 4; }

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

int pick_router_bn(int E) {
  if (E <= 16) return 16;
  if (E <= 32) return 32;
  if (E <= 64) return 64;
  if (E <= 128) return 128;
  return 256;
}

// Split-K factor of the tensor-core router GEMM: enough CTAs to stream x at HBM speed when
// T/128 row tiles alone would leave most SMs idle. A function of the shape only (148 is the
// B300 SM count), so the summation order -- and every bit of the logits -- is fixed.
struct RouterSplit {
  int splits, kb_per_split;
};
RouterSplit router_split(const moe_shape* s) {
  if (s->dtype != MOE_BF16 || s->T == 0) return {1, 0};
  const int bn = pick_router_bn(s->E);
  const long long tiles = static_cast<long long>((s->T + 127) / 128) * ((s->E + bn - 1) / bn);
  const int nk = (s->d + 63) / 64;
  long long want = 148 / std::max<long long>(tiles, 1);
  want = std::max<long long>(1, std::min<long long>(want, std::min(16, nk)));
  const int kb = (nk + static_cast<int>(want) - 1) / static_cast<int>(want);
  return {(nk + kb - 1) / kb, kb};
}

bool expert_choice(const moe_shape* s) { return s->gate == MOE_GATE_EXPERT_CHOICE; }

// bf16 layers with E <= 256 route from x with the fused router (router_fused.cu: logits on
// chip, split-K partials reduced in a cluster); others run the router GEMM into split-K logit
// planes and the top-k kernel on them.
bool fused_router(const moe_shape* s) {
  return s->dtype == MOE_BF16 && s->E <= 256 && s->T > 0;
}

// Per-block statistic partials the routing step writes from x (fused router: one per CTA),
// and the most any routing call writes (the workspace holds that many).
int route_partials_from_x(const moe_shape* s) {
  return fused_router(s) ? router_fused_plan(s->T, s->d, s->E).grid : route_blocks(s->T);
}
int route_partial_blocks(const moe_shape* s) {
  return std::max(route_blocks(s->T), route_partials_from_x(s));
}

// Rows of the permuted activations: T*k assignments, or E*min(C, T) for expert choice.
size_t perm_rows(const moe_shape* s) {
  if (expert_choice(s))
    return static_cast<size_t>(s->E) * static_cast<size_t>(std::min(s->capacity, s->T));
  return static_cast<size_t>(s->T) * s->k;
}

struct Layout {
  size_t err, logits, idx, gate, partials, stats, counts, offsets, perm, inv, dropped, losses,
      blk_hist, probs;
  size_t xp, h, yp, hs, ys, total;
};

Layout layout(const moe_shape* s) {
  const size_t T = s->T, E = s->E, k = s->k, d = s->d, F = s->d_ff, Fs = s->d_ff_shared;
  const size_t es = esize(s);
  const size_t A = T * k;
  const size_t R = perm_rows(s);
  const bool ec = expert_choice(s);
  Layout L;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + std::max<size_t>(bytes, 1));
    return at;
  };
  L.err = take(sizeof(DeviceError));
  L.logits = take(static_cast<size_t>(router_split(s).splits) * T * E * 4);
  L.idx = take(A * 4);
  L.gate = take(std::max(A, R) * 4);
  L.partials = take(static_cast<size_t>(route_partial_blocks(s)) * (E + 1) * 4);
  L.stats = take((E + 1) * 4);
  L.counts = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.perm = take(std::max(A, R) * 4);
  L.inv = take(ec ? T * E * 4 : A * 4);
  L.dropped = take(4);
  L.losses = take(2 * 4);
  L.blk_hist = take(static_cast<size_t>(dispatch_max_blocks(148)) * E * 4);
  L.probs = take(ec ? T * E * 4 : 0);
  L.xp = take(R * d * es);
  L.h = take(R * F * es);
  L.yp = take(R * d * es);
  L.hs = take(Fs > 0 ? T * Fs * es : 0);
  L.ys = take(Fs > 0 ? T * d * es : 0);
  L.total = o;
  return L;
}

int check_shape(const moe_shape* s) {
  if (s == nullptr) return fail(MOE_ERR_INVALID, "shape is NULL");
  if (s->T < 0) return fail(MOE_ERR_INVALID, "T = %d < 0", s->T);
  if (s->d < 1) return fail(MOE_ERR_INVALID, "d = %d < 1", s->d);
  if (s->E < 1 || s->E > 1024) return fail(MOE_ERR_INVALID, "E = %d outside 1..1024", s->E);
  if (s->k < 1 || s->k > s->E) return fail(MOE_ERR_INVALID, "k = %d outside 1..E (E = %d)", s->k, s->E);
  if (s->d_ff < 1) return fail(MOE_ERR_INVALID, "d_ff = %d < 1", s->d_ff);
  if (s->d_ff_shared < 0) return fail(MOE_ERR_INVALID, "d_ff_shared = %d < 0", s->d_ff_shared);
  if (s->capacity < 0) return fail(MOE_ERR_INVALID, "capacity = %d < 0", s->capacity);
  if (s->gate < MOE_GATE_SOFTMAX_ALL || s->gate > MOE_GATE_EXPERT_CHOICE)
    return fail(MOE_ERR_INVALID, "gate mode %d unknown", s->gate);
  if (s->dtype != MOE_F32 && s->dtype != MOE_BF16)
    return fail(MOE_ERR_INVALID, "dtype %d unknown", s->dtype);
  if (static_cast<long long>(s->T) * s->k >= (1ll << 31))
    return fail(MOE_ERR_INVALID, "T*k = %lld does not fit int32", static_cast<long long>(s->T) * s->k);
  if (s->gate == MOE_GATE_EXPERT_CHOICE &&
      static_cast<long long>(s->T) * s->E >= (1ll << 31))
    return fail(MOE_ERR_INVALID, "expert choice needs T*E < 2^31");
  if ((static_cast<size_t>(s->d) * esize(s)) % 16 != 0)
    return fail(MOE_ERR_UNSUPPORTED, "d * sizeof(dtype) = %zu is not a multiple of 16 bytes",
                static_cast<size_t>(s->d) * esize(s));
  if (s->dtype == MOE_BF16 && (s->d_ff % 8 != 0 || s->d_ff_shared % 8 != 0))
    return fail(MOE_ERR_UNSUPPORTED, "bf16 needs d_ff and d_ff_shared multiples of 8");
  if (s->dtype == MOE_F32 && ((s->T + 31) / 32 > 65535))
    return fail(MOE_ERR_UNSUPPORTED, "fp32 path supports T <= %d", 65535 * 32);
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

#define REQUIRE_PTR(p, name)                                                 \
  do {                                                                       \
    if ((p) == nullptr) return fail(MOE_ERR_INVALID, "%s is NULL", name);    \
    if (!aligned16(p)) return fail(MOE_ERR_INVALID, "%s is not 16-byte aligned", name); \
  } while (0)
#define REQUIRE_PTR4(p, name)                                                \
  do {                                                                       \
    if ((p) == nullptr) return fail(MOE_ERR_INVALID, "%s is NULL", name);    \
    if (!aligned4(p)) return fail(MOE_ERR_INVALID, "%s is not 4-byte aligned", name); \
  } while (0)
#define OPT_PTR4(p, name)                                                    \
  do {                                                                       \
    if ((p) != nullptr && !aligned4(p))                                      \
      return fail(MOE_ERR_INVALID, "%s is not 4-byte aligned", name);        \
  } while (0)
#define TRY(expr)                       \
  do {                                  \
    const int rc_ = (expr);             \
    if (rc_ != MOE_OK) return rc_;      \
  } while (0)

int check_ws(const moe_shape* s, const void* ws, size_t ws_bytes) {
  if (ws == nullptr) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0)
    return fail(MOE_ERR_WORKSPACE, "workspace is not %zu-byte aligned", kAlign);
  const size_t need = layout(s).total;
  if (ws_bytes < need)
    return fail(MOE_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  return MOE_OK;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return n;
}

int cuda_status(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return MOE_OK;
}

#define LAUNCH(expr, what)                                                   \
  do {                                                                       \
    const int rc_ = (expr);                                                  \
    if (rc_ != MOE_OK) {                                                     \
      if (rc_ == MOE_ERR_CUDA) return cuda_status(what);                     \
      return fail(rc_, "%s failed", what);                                   \
    }                                                                        \
  } while (0)

// ---------------------------------------------------------------- stage 0: router GEMM
// Writes router_split(s).splits partial logit planes [T, E] (fp32, no bias) to `logits`.
int run_router(const moe_shape* s, const void* x, const void* wr, float* logits, DeviceError* err,
               cudaStream_t st) {
  if (s->T == 0) return MOE_OK;
  if (s->dtype == MOE_F32) {
    SimtArgs a{};
    a.groups = 1;
    a.offsets = nullptr;
    a.m_single = s->T;
    a.max_rows = s->T;
    a.a = static_cast<const float*>(x);
    a.b0 = static_cast<const float*>(wr);
    a.n = s->E;
    a.k = s->d;
    a.out = logits;
    a.bias = nullptr;  // added by the top-k kernel
    LAUNCH(launch_simt_gemm(TC_F32OUT, a, st), "router GEMM (fp32)");
    return MOE_OK;
  }
  const int bn = pick_router_bn(s->E);
  const RouterSplit sp = router_split(s);
  TcProblem p{};
  p.args.groups = 1;
  p.args.offsets = nullptr;
  p.args.m_single = s->T;
  p.args.n_routed = s->E;
  p.args.k_routed = s->d;
  p.args.out_routed = logits;
  p.args.ldo_routed = s->E;
  p.args.bias = nullptr;  // added by the top-k kernel, after the split-K sum
  p.args.splits = sp.splits;
  p.args.kb_per_split = sp.kb_per_split;
  p.args.split_stride = static_cast<long long>(s->T) * s->E;
  p.args.err = err;
  p.a = x;
  p.a_rows = s->T;
  p.b0 = wr;
  p.b_rows = s->E;
  p.b_groups = 1;
  p.max_tiles = static_cast<long long>((s->T + 127) / 128) * ((s->E + bn - 1) / bn) * sp.splits;
  p.num_sms = num_sms();
  LAUNCH(launch_tc_gemm(TC_F32OUT, bn, 1, 64, false, 128, p, st), "router GEMM (tcgen05)");
  return MOE_OK;
}

RouteArgs route_args(const moe_shape* s, const float* logits, int nsplit, const float* bias,
                     float* logits_out, int32_t* idx, float* gate, float* partials,
                     DeviceError* err, const float* select_bias = nullptr) {
  RouteArgs a{};
  a.logits = logits;
  a.nsplit = nsplit;
  a.split_stride = static_cast<size_t>(s->T) * s->E;
  a.bias = bias;
  a.select_bias = select_bias;
  a.logits_out = logits_out;
  a.T = s->T;
  a.E = s->E;
  a.k = s->k;
  a.gate_mode = s->gate;
  a.topk_idx = idx;
  a.topk_gate = gate;
  a.partials = partials;
  a.err = err;
  return a;
}

// Steps 1-2 from x: the logits, then the routing step `ra` (its logits / nsplit fields are
// set here). Records `ev_mid` (if any) between the logits and the routing step: with the
// fused router both are one kernel, so the event follows it. Writes
// route_partials_from_x(s) statistic partials.
int route_from_x(const moe_shape* s, const void* x, const void* wr, RouteArgs ra, float* planes,
                 DeviceError* err, cudaStream_t st, cudaEvent_t ev_mid = nullptr) {
  if (s->T == 0) {
    if (ev_mid) cudaEventRecord(ev_mid, st);
    return MOE_OK;
  }
  if (fused_router(s)) {
    LAUNCH(launch_router_fused(router_fused_plan(s->T, s->d, s->E), x, wr, ra, s->d, st),
           "router with fused gates/top-k");
    if (ev_mid) cudaEventRecord(ev_mid, st);
    return MOE_OK;
  }
  TRY(run_router(s, x, wr, planes, err, st));
  if (ev_mid) cudaEventRecord(ev_mid, st);
  ra.logits = planes;
  ra.nsplit = router_split(s).splits;
  ra.split_stride = static_cast<size_t>(s->T) * s->E;
  LAUNCH(launch_route_topk(ra, st), "gates/top-k");
  return MOE_OK;
}

// ---------------------------------------------------------------- stages 4-5: expert GEMMs
// 8-bit expert weights: E4M3 codes [E, rows, K] and one fp32 scale per row [E, rows].
struct Fp8Weights {
  const uint8_t *w1q, *w3q, *w2q;
  const float *w1s, *w3s, *w2s;
};

int check_fp8(const moe_shape* s, const Fp8Weights* q) {
  if (s->dtype != MOE_BF16) return fail(MOE_ERR_UNSUPPORTED, "8-bit weights need a bf16 layer");
  if (s->d_ff_shared != 0)
    return fail(MOE_ERR_UNSUPPORTED, "8-bit weights: no shared expert supported");
  if (s->d % 16 != 0 || s->d_ff % 16 != 0)
    return fail(MOE_ERR_UNSUPPORTED, "8-bit weights need d and d_ff multiples of 16");
  REQUIRE_PTR(q->w1q, "w1q");
  REQUIRE_PTR(q->w3q, "w3q");
  REQUIRE_PTR(q->w2q, "w2q");
  REQUIRE_PTR4(q->w1s, "w1_scale");
  REQUIRE_PTR4(q->w3s, "w3_scale");
  REQUIRE_PTR4(q->w2s, "w2_scale");
  return MOE_OK;
}

// Top-1 bf16 layers without a shared expert (and not expert choice) need no combine: the
// down projection's epilogue writes g * (H W2^T) of row r straight to y[perm[r]], and the
// gather zeroes the rows of dropped tokens.
bool combine_in_epilogue(const moe_shape* s) {
  return s->k == 1 && !expert_choice(s) && s->d_ff_shared == 0 && s->dtype == MOE_BF16;
}

// Expert-choice layers pass row_gate (gate per row) and perm holding token indices; top-k
// layers pass gate (per assignment, looked up through perm) and perm holding assignments.
// q != nullptr: the routed expert weights are 8-bit (w1/w3/w2 are ignored).
// inv and y non-null (combine_in_epilogue layers, bf16 weights): the layer's output is
// written here directly (y_perm unused).
int run_experts(const moe_shape* s, const void* x, const int32_t* perm, const int32_t* offsets,
                const float* gate, const float* row_gate, const void* w1, const void* w3,
                const void* w2, const void* w1s, const void* w3s, const void* w2s, void* y_perm,
                void* y_shared, void* ws, cudaStream_t st, void* const* ev, int ev_first,
                const Fp8Weights* q = nullptr, const int32_t* inv = nullptr, void* y = nullptr) {
  const bool direct = inv != nullptr && y != nullptr;
  if (direct && (!combine_in_epilogue(s) || q != nullptr || gate == nullptr))
    return fail(MOE_ERR_INVALID, "direct output needs a top-1 bf16 layer");
  const Layout L = layout(s);
  DeviceError* err = at<DeviceError>(ws, L.err);
  const int A = static_cast<int>(perm_rows(s));
  const int gather_k = expert_choice(s) ? 1 : s->k;
  const bool shared = s->d_ff_shared > 0;
  void* xp = at<void>(ws, L.xp);
  void* h = at<void>(ws, L.h);
  void* hs = at<void>(ws, L.hs);
  const int sms = num_sms();
  const int max_group_rows = std::min(s->T, s->capacity);

  auto rec = [&](int i) {
    if (ev && ev[i]) cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), st);
  };

  // stage 3: gather
  rec(ev_first);
  if (direct)
    LAUNCH(launch_gather_tokens(x, inv, s->T, static_cast<int>(s->d * esize(s)), xp, y, sms, st),
           "gather (token-major)");
  else
    LAUNCH(launch_gather(x, perm, offsets, s->E, gather_k, static_cast<int>(s->d * esize(s)), A,
                         xp, sms, st, q != nullptr ? err : nullptr),
           "gather");

  if (s->dtype == MOE_F32) {
    rec(ev_first + 1);
    SimtArgs g1{};
    g1.groups = s->E;
    g1.offsets = offsets;
    g1.max_rows = max_group_rows;
    g1.a = static_cast<const float*>(xp);
    g1.b0 = static_cast<const float*>(w1);
    g1.b1 = static_cast<const float*>(w3);
    g1.n = s->d_ff;
    g1.k = s->d;
    g1.out = static_cast<float*>(h);
    LAUNCH(launch_simt_gemm(TC_SWIGLU, g1, st), "gate/up GEMM (fp32)");
    if (shared) {
      SimtArgs gs = g1;
      gs.groups = 1;
      gs.offsets = nullptr;
      gs.m_single = s->T;
      gs.max_rows = s->T;
      gs.a = static_cast<const float*>(x);
      gs.b0 = static_cast<const float*>(w1s);
      gs.b1 = static_cast<const float*>(w3s);
      gs.n = s->d_ff_shared;
      gs.out = static_cast<float*>(hs);
      LAUNCH(launch_simt_gemm(TC_SWIGLU, gs, st), "shared gate/up GEMM (fp32)");
    }
    rec(ev_first + 2);
    SimtArgs g2{};
    g2.groups = s->E;
    g2.offsets = offsets;
    g2.max_rows = max_group_rows;
    g2.a = static_cast<const float*>(h);
    g2.b0 = static_cast<const float*>(w2);
    g2.n = s->d;
    g2.k = s->d_ff;
    g2.out = static_cast<float*>(y_perm);
    g2.perm = perm;
    g2.gate = gate;
    g2.row_gate = row_gate;
    LAUNCH(launch_simt_gemm(TC_SCALE, g2, st), "down GEMM (fp32)");
    if (shared) {
      SimtArgs gs = g2;
      gs.groups = 1;
      gs.offsets = nullptr;
      gs.m_single = s->T;
      gs.max_rows = s->T;
      gs.a = static_cast<const float*>(hs);
      gs.b0 = static_cast<const float*>(w2s);
      gs.k = s->d_ff_shared;
      gs.out = static_cast<float*>(y_shared);
      gs.perm = nullptr;
      gs.gate = nullptr;
      gs.row_gate = nullptr;
      LAUNCH(launch_simt_gemm(TC_SCALE, gs, st), "shared down GEMM (fp32)");
    }
    return MOE_OK;
  }

  // bf16: tcgen05 grouped GEMMs, routed experts and the shared expert in one launch each.
  // The kernel is bound by load latency: 256-row CTA tiles (one weight tile feeds two MMAs,
  // twice the MMA work per staged byte) hide more of it, but fill TMEM, so their epilogue is
  // not double-buffered, and they pull every weight tile from DRAM in one CTA instead of
  // sharing it through L2 with a neighbour. They win when experts average >= 512 rows (and,
  // for the down projection, with its lighter epilogue, when d_ff >= 8192); otherwise
  // 128-row tiles with double-buffered accumulators.
  const long long kept_max = std::min<long long>(A, static_cast<long long>(s->E) * max_group_rows);
  const bool w8 = q != nullptr;  // 8-bit weights: 128-row tiles only
  const bool mt2_ok = !w8 && s->E <= kTcMt2MaxGroups && kept_max / s->E >= 512;
  const int mt_gateup = mt2_ok ? 2 : 1;
  const int mt_down = (mt2_ok && s->d_ff >= 8192) ? 2 : 1;
  // 256-row tiles on CTA pairs (tc_pair.cu): both halves' accumulators double-buffered, but
  // a pair always multiplies 256 rows, where a single CTA skips the empty second half of a
  // group's last tile. So pairs only where the host knows every group's size and the last
  // tile is more than half full: expert-choice layers, each expert holding min(C, T) rows.
  const int ec_rows = std::min(s->capacity, s->T);
  const bool pair_tiles = expert_choice(s) && (ec_rows % 256 == 0 || ec_rows % 256 > 128);
  const int kb_gateup = 64, kb_down = 64;
  // Gate/up MMA width with 128-row tiles: 256 (128 H columns per tile) or 224 (112), which
  // ever leaves fewer SMs idle in the last wave of the estimated tile count (e.g. the
  // Mixtral-shaped decode step: 896 tiles = 6.05 waves at 256, 1024 = 6.92 waves at 224).
  int bn_gateup = 256;
  if (mt_gateup == 1 && s->d_ff % 112 == 0) {
    const long long rows_e = std::max<long long>(1, (kept_max + s->E - 1) / s->E);
    const long long row_tiles_est = ((rows_e + 127) / 128) * s->E;
    auto wave_eff = [&](int bn_out) {
      const long long tiles = row_tiles_est * ((s->d_ff + bn_out - 1) / bn_out);
      const long long rounds = (tiles + sms - 1) / sms;
      return static_cast<double>(tiles) / static_cast<double>(rounds * sms);
    };
    if (wave_eff(112) > wave_eff(128) + 0.02) bn_gateup = 224;
  }
  // Short row tiles (32 rows of A per k-block instead of 128) when no group has more than
  // 32 rows, e.g. a decode step: a quarter of the A bytes per stage, so more stages and
  // more weight bytes in flight.
  const int ar = (mt_gateup == 1 && mt_down == 1 && (shared ? s->T : max_group_rows) <= 32)
                     ? 32 : 128;
  auto row_tiles = [&](int mt, long long rows) {
    const int tm = ar < 128 ? ar : 128 * mt;
    return (rows + tm - 1) / tm;
  };

  rec(ev_first + 1);
  {
    TcProblem p{};
    p.args.groups = s->E;
    p.args.offsets = offsets;
    p.args.n_routed = s->d_ff;
    p.args.k_routed = s->d;
    p.args.out_routed = h;
    p.args.ldo_routed = s->d_ff;
    if (w8) {
      p.args.scale0 = q->w1s;
      p.args.scale1 = q->w3s;
    }
    p.args.has_shared = shared;
    p.args.m_shared = s->T;
    p.args.n_shared = s->d_ff_shared;
    p.args.k_shared = s->d;
    p.args.out_shared = hs;
    p.args.ldo_shared = s->d_ff_shared;
    p.args.err = err;
    p.a = xp;
    p.a_rows = std::max(A, 1);
    p.b0 = w8 ? static_cast<const void*>(q->w1q) : w1;
    p.b1 = w8 ? static_cast<const void*>(q->w3q) : w3;
    p.b_rows = s->d_ff;
    p.b_groups = s->E;
    p.a_s = x;
    p.b0_s = w1s;
    p.b1_s = w3s;
    p.b_rows_s = s->d_ff_shared;
    const int bno = bn_gateup / 2;
    p.max_tiles = (row_tiles(mt_gateup, kept_max) + s->E) * ((s->d_ff + bno - 1) / bno) +
                  (shared ? row_tiles(mt_gateup, s->T) * ((s->d_ff_shared + bno - 1) / bno) : 0);
    p.num_sms = sms;
    if (mt_gateup == 2 && pair_tiles)
      LAUNCH(launch_tc_pair_gemm(TC_SWIGLU, p, st), "gate/up GEMM (tcgen05, CTA pairs)");
    else
      LAUNCH(launch_tc_gemm(TC_SWIGLU, bn_gateup, mt_gateup, kb_gateup, w8, ar, p, st),
           "gate/up GEMM (tcgen05)");
  }
  rec(ev_first + 2);
  {
    TcProblem p{};
    p.args.groups = s->E;
    p.args.offsets = offsets;
    p.args.n_routed = s->d;
    p.args.k_routed = s->d_ff;
    p.args.out_routed = direct ? y : y_perm;
    p.args.ldo_routed = s->d;
    p.args.scatter_rows = direct ? 1 : 0;
    if (w8) p.args.scale0 = q->w2s;
    p.args.has_shared = shared;
    p.args.m_shared = s->T;
    p.args.n_shared = s->d;
    p.args.k_shared = s->d_ff_shared;
    p.args.out_shared = y_shared;
    p.args.ldo_shared = s->d;
    p.args.perm = perm;
    p.args.gate = gate;
    p.args.row_gate = row_gate;
    p.args.err = err;
    p.a = h;
    p.a_rows = std::max(A, 1);
    p.b0 = w8 ? static_cast<const void*>(q->w2q) : w2;
    p.b_rows = s->d;
    p.b_groups = s->E;
    p.a_s = hs;
    p.b0_s = w2s;
    p.b_rows_s = s->d;
    const int bn = 256;
    p.max_tiles = (row_tiles(mt_down, kept_max) + s->E + (shared ? row_tiles(mt_down, s->T) : 0)) *
                  ((s->d + bn - 1) / bn);
    p.num_sms = sms;
    if (mt_down == 2 && pair_tiles)
      LAUNCH(launch_tc_pair_gemm(TC_SCALE, p, st), "down GEMM (tcgen05, CTA pairs)");
    else
      LAUNCH(launch_tc_gemm(TC_SCALE, bn, mt_down, kb_down, w8, ar, p, st), "down GEMM (tcgen05)");
  }
  return MOE_OK;
}

// ---------------------------------------------------------------- block-scaled experts
// Weights as E4M3 codes (fmt MOE_MX_E4M3) or E2M1 codes packed two per byte (MOE_MX_E2M1),
// each with its scale atoms (tc_mx.cu).
struct MxWeights {
  int fmt;
  const uint8_t *w1q, *w3q, *w2q;
  const uint8_t *w1sf, *w3sf, *w2sf;
};

// The forward's layout, then the block-scaled operands: the gathered x rows as E4M3 codes
// [R, d] with their scale atoms, and the hidden rows H as E4M3 codes [R, d_ff] with theirs.
// Row tiles: at most R / 32 + E + 1 (32-row tiles; each expert adds at most one partial tile).
struct MxLayout {
  Layout f;
  size_t xq, xsf, hq, hsf, total;
};

MxLayout layout_mx(const moe_shape* s) {
  MxLayout M;
  M.f = layout(s);
  const size_t R = perm_rows(s), d = s->d, F = s->d_ff;
  const size_t tiles = R / 32 + static_cast<size_t>(s->E) + 1;
  size_t o = M.f.total;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + std::max<size_t>(bytes, 1));
    return at;
  };
  M.xq = take(R * d);
  M.xsf = take(tiles * (d / 128) * 512);
  M.hq = take(R * F);
  M.hsf = take(tiles * (F / 128) * 512);
  M.total = o;
  return M;
}

int check_mx_shape(const moe_shape* s, int fmt) {
  if (fmt != MOE_MX_E4M3 && fmt != MOE_MX_E2M1)
    return fail(MOE_ERR_INVALID, "block-scaled weight format %d unknown", fmt);
  if (s->dtype != MOE_BF16)
    return fail(MOE_ERR_UNSUPPORTED, "block-scaled weights need a bf16 layer");
  if (s->d_ff_shared != 0)
    return fail(MOE_ERR_UNSUPPORTED, "block-scaled weights: no shared expert supported");
  if (expert_choice(s))
    return fail(MOE_ERR_UNSUPPORTED, "block-scaled weights: top-k routing only");
  if (s->d % 256 != 0 || s->d_ff % 128 != 0)
    return fail(MOE_ERR_UNSUPPORTED,
                "block-scaled weights need d a multiple of 256 and d_ff a multiple of 128");
  return MOE_OK;
}

bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

int check_mx(const moe_shape* s, const MxWeights* m) {
  TRY(check_mx_shape(s, m->fmt));
  const uint8_t* q[3] = {m->w1q, m->w3q, m->w2q};
  const uint8_t* sf[3] = {m->w1sf, m->w3sf, m->w2sf};
  const char* qn[3] = {"w1q", "w3q", "w2q"};
  const char* sn[3] = {"w1_scales", "w3_scales", "w2_scales"};
  for (int i = 0; i < 3; ++i) {
    REQUIRE_PTR(q[i], qn[i]);
    if (m->fmt == MOE_MX_E2M1 && !aligned32(q[i]))
      return fail(MOE_ERR_INVALID, "%s (4-bit codes) is not 32-byte aligned", qn[i]);
    REQUIRE_PTR(sf[i], sn[i]);
  }
  return MOE_OK;
}

// Stages 3-5 on block-scaled experts: gather + quantize x, gate/up GEMM writing H as
// block-scaled E4M3, down GEMM writing g * (H . W2^T) as bf16 rows.
int run_experts_mx(const moe_shape* s, const void* x, const int32_t* perm, const int32_t* offsets,
                   const float* gate, const MxWeights* m, void* y_perm, void* ws, cudaStream_t st,
                   void* const* ev, int ev_first) {
  const MxLayout M = layout_mx(s);
  DeviceError* err = at<DeviceError>(ws, M.f.err);
  const long long A = static_cast<long long>(perm_rows(s));
  const int sms = num_sms();
  const int max_group_rows = std::min(s->T, s->capacity);
  const int ar = max_group_rows <= 32 ? 32 : 128;
  const int bfmt = m->fmt == MOE_MX_E2M1 ? 5 : 0;
  const long long kept_max = std::min<long long>(A, static_cast<long long>(s->E) * max_group_rows);
  const long long row_tiles = (kept_max + ar - 1) / ar + s->E;
  uint8_t* xq = at<uint8_t>(ws, M.xq);
  uint8_t* xsf = at<uint8_t>(ws, M.xsf);
  uint8_t* hq = at<uint8_t>(ws, M.hq);
  uint8_t* hsf = at<uint8_t>(ws, M.hsf);
  auto rec = [&](int i) {
    if (ev && ev[i]) cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), st);
  };

  rec(ev_first);
  LAUNCH(launch_mx_gather_quant(x, perm, offsets, s->E, s->k, s->d, ar, A, xq, xsf, err, sms, st),
         "gather + block quantization");
  rec(ev_first + 1);
  {
    MxProblem p{};
    p.args.groups = s->E;
    p.args.offsets = offsets;
    p.args.n = s->d_ff;
    p.args.n_rows = s->d_ff;
    p.args.k = s->d;
    p.args.sfa = xsf;
    p.args.sfb0 = m->w1sf;
    p.args.sfb1 = m->w3sf;
    p.args.out_codes = hq;
    p.args.out_atoms = hsf;
    p.args.err = err;
    p.a = xq;
    p.a_rows = std::max(A, 1ll);
    p.b0 = m->w1q;
    p.b1 = m->w3q;
    p.max_tiles = row_tiles * (s->d_ff / 128);
    p.num_sms = sms;
    LAUNCH(launch_mx_gemm(TC_SWIGLU, ar, bfmt, p, st), "gate/up GEMM (block-scaled)");
  }
  rec(ev_first + 2);
  {
    MxProblem p{};
    p.args.groups = s->E;
    p.args.offsets = offsets;
    p.args.n = s->d;
    p.args.n_rows = s->d;
    p.args.k = s->d_ff;
    p.args.sfa = hsf;
    p.args.sfb0 = m->w2sf;
    p.args.out_rows = y_perm;
    p.args.ldo = s->d;
    p.args.perm = perm;
    p.args.gate = gate;
    p.args.err = err;
    p.a = hq;
    p.a_rows = std::max(A, 1ll);
    p.b0 = m->w2q;
    p.max_tiles = row_tiles * (s->d / 256);
    p.num_sms = sms;
    LAUNCH(launch_mx_gemm(TC_SCALE, ar, bfmt, p, st), "down GEMM (block-scaled)");
  }
  return MOE_OK;
}

// Every argument check of the layer's forward, made on the host before anything is queued.
int check_forward(const moe_shape* s, const void* x, const void* w_router, const float* router_bias,
                  const void* w1, const void* w3, const void* w2, const void* w1s, const void* w3s,
                  const void* w2s, const void* y, const int32_t* counts, const int32_t* dropped,
                  const float* losses, const void* ws, size_t ws_bytes, void* const* ev, int n_ev,
                  const Fp8Weights* q, const MxWeights* mx = nullptr) {
  TRY(check_shape(s));
  if (mx != nullptr) {
    TRY(check_mx(s, mx));
    TRY(check_ws(s, ws, ws_bytes));
    const size_t need = layout_mx(s).total;
    if (ws_bytes < need)
      return fail(MOE_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu (moe_mx_workspace_size)",
                  ws_bytes, need);
  } else {
    TRY(check_ws(s, ws, ws_bytes));
  }
  if (q != nullptr) TRY(check_fp8(s, q));
  if (ev != nullptr && n_ev != MOE_NUM_STAGES + 1)
    return fail(MOE_ERR_INVALID, "n_events = %d, expected %d", n_ev, MOE_NUM_STAGES + 1);
  if (s->T > 0) {
    REQUIRE_PTR(x, "x");
    REQUIRE_PTR(w_router, "w_router");
    if (q == nullptr && mx == nullptr) {
      REQUIRE_PTR(w1, "w1");
      REQUIRE_PTR(w3, "w3");
      REQUIRE_PTR(w2, "w2");
    }
    REQUIRE_PTR(y, "y");
    if (s->d_ff_shared > 0) {
      REQUIRE_PTR(w1s, "w1s");
      REQUIRE_PTR(w3s, "w3s");
      REQUIRE_PTR(w2s, "w2s");
    }
  }
  OPT_PTR4(router_bias, "router_bias");
  OPT_PTR4(counts, "counts");
  OPT_PTR4(dropped, "dropped");
  OPT_PTR4(losses, "losses");
  return MOE_OK;
}

int forward_impl(const moe_shape* s, const void* x, const void* w_router, const float* router_bias,
                 const void* w1, const void* w3, const void* w2, const void* w1s, const void* w3s,
                 const void* w2s, void* y, int32_t* counts, int32_t* dropped, float* losses,
                 void* ws, size_t ws_bytes, void* stream, void* const* ev, int n_ev,
                 float* select_bias = nullptr, float gamma = 0.f,
                 const Fp8Weights* q = nullptr, const MxWeights* mx = nullptr) {
  TRY(check_forward(s, x, w_router, router_bias, w1, w3, w2, w1s, w3s, w2s, y, counts, dropped,
                    losses, ws, ws_bytes, ev, n_ev, q, mx));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Layout L = layout(s);
  DeviceError* err = at<DeviceError>(ws, L.err);
  float* logits = at<float>(ws, L.logits);
  int32_t* idx = at<int32_t>(ws, L.idx);
  float* gate = at<float>(ws, L.gate);
  float* partials = at<float>(ws, L.partials);
  float* stats = at<float>(ws, L.stats);
  int32_t* cnt = counts ? counts : at<int32_t>(ws, L.counts);
  int32_t* off = at<int32_t>(ws, L.offsets);
  int32_t* perm = at<int32_t>(ws, L.perm);
  int32_t* inv = at<int32_t>(ws, L.inv);
  int32_t* drp = dropped ? dropped : at<int32_t>(ws, L.dropped);
  float* los = losses ? losses : at<float>(ws, L.losses);
  void* yp = at<void>(ws, L.yp);
  void* ys = s->d_ff_shared > 0 ? at<void>(ws, L.ys) : nullptr;
  auto rec = [&](int i) {
    if (ev && ev[i]) cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), st);
  };

  const bool ec = expert_choice(s);
  if (ec && select_bias != nullptr)
    return fail(MOE_ERR_UNSUPPORTED, "selection bias applies to top-k routing only");
  rec(0);
  {
    RouteArgs ra = route_args(s, nullptr, 1, router_bias, nullptr, idx, gate, partials, err,
                              select_bias);
    if (ec) {
      ra.k = 0;  // probabilities and statistics only; the experts choose below
      ra.probs_t = at<float>(ws, L.probs);
    }
    TRY(route_from_x(s, x, w_router, ra, logits, err, st,
                     ev ? static_cast<cudaEvent_t>(ev[1]) : nullptr));
  }
  rec(2);
  if (ec) {
    LAUNCH(launch_expert_choice(at<float>(ws, L.probs), s->T, s->E, s->capacity, perm, gate, inv,
                                cnt, off, drp, st),
           "expert choice");
  } else {
    // the statistics and losses ride along in one more CTA of the dispatch
    DispatchLoss dl{partials, route_partials_from_x(s), stats, s->T, s->k, s->alpha, s->beta, los};
    LAUNCH(launch_dispatch(idx, s->T * s->k, s->E, s->capacity, cnt, off, perm, inv, drp,
                           at<int32_t>(ws, L.blk_hist), err, num_sms(), st,
                           s->T > 0 ? &dl : nullptr),
           "dispatch (with the router statistics and losses)");
  }
  // top-1 bf16 layers: the down projection writes y itself (no combine launch)
  const bool direct = combine_in_epilogue(s) && q == nullptr && mx == nullptr;
  if (s->T > 0 && mx != nullptr) {
    TRY(run_experts_mx(s, x, perm, off, gate, mx, yp, ws, st, ev, 3));
  } else if (s->T > 0) {
    TRY(run_experts(s, x, perm, off, ec ? nullptr : gate, ec ? gate : nullptr, w1, w3, w2, w1s,
                    w3s, w2s, yp, ys, ws, st, ev, 3, q, direct ? inv : nullptr,
                    direct ? y : nullptr));
  } else {
    rec(3);
    rec(4);
    rec(5);
  }
  rec(6);
  if (!direct)
    LAUNCH(launch_combine(s->dtype, yp, inv, ys, y, s->T, ec ? s->E : s->k, s->d, num_sms(), st),
           "combine");
  rec(7);
  if (s->T > 0) {
    if (ec)
      LAUNCH(launch_stats_loss(partials, route_partials_from_x(s), s->E, stats, cnt, s->T, s->k,
                               s->alpha, s->beta, los, err, st),
             "router statistics and losses");
  } else {
    LAUNCH(launch_aux_loss(stats, cnt, s->T, s->E, s->k, s->alpha, s->beta, los, st), "aux loss");
  }
  if (select_bias != nullptr)
    LAUNCH(launch_update_select_bias(cnt, select_bias, s->T, s->E, s->k, gamma, st),
           "selection bias update");
  rec(8);
  return ok();
}

}  // namespace

int set_error_detail(int status, const char* text) {
  g_detail = text;
  return status;
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_capacity(double cf, int32_t T, int32_t k, int32_t E) {
  if (E < 1 || k < 1 || T < 0 || !(cf >= 0.0)) return -1;
  const double c = std::ceil(cf * static_cast<double>(T) * static_cast<double>(k) /
                             static_cast<double>(E));
  if (c >= static_cast<double>(T)) return T;
  return static_cast<int>(c);
}

int moe_check_shape(const moe_shape* s) {
  const int rc = check_shape(s);
  return rc == MOE_OK ? ok() : rc;
}

size_t moe_workspace_size(const moe_shape* s) {
  if (check_shape(s) != MOE_OK) return 0;
  return layout(s).total;
}

}  // extern "C"

namespace {
int route_impl(const moe_shape* s, const void* x, const void* w_router, const float* router_bias,
               const float* logits_in, const float* select_bias, float* logits_out,
               int32_t* topk_idx, float* topk_gate, float* stats, void* ws, size_t ws_bytes,
               void* stream) {
  TRY(check_shape(s));
  if (expert_choice(s))
    return fail(MOE_ERR_UNSUPPORTED, "expert-choice layers route with moe_expert_choice");
  TRY(check_ws(s, ws, ws_bytes));
  if (s->T > 0) {
    if (logits_in == nullptr) {
      REQUIRE_PTR(x, "x");
      REQUIRE_PTR(w_router, "w_router");
      OPT_PTR4(router_bias, "router_bias");
    } else {
      REQUIRE_PTR4(logits_in, "logits_in");
    }
    REQUIRE_PTR4(topk_idx, "topk_idx");
    REQUIRE_PTR4(topk_gate, "topk_gate");
  }
  OPT_PTR4(logits_out, "logits_out");
  OPT_PTR4(stats, "stats");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Layout L = layout(s);
  DeviceError* err = at<DeviceError>(ws, L.err);
  if (s->T == 0) {
    if (stats && cudaMemsetAsync(stats, 0, (s->E + 1) * sizeof(float), st) != cudaSuccess)
      return cuda_status("memset stats");
    return ok();
  }
  float* partials = at<float>(ws, L.partials);
  int nb = route_blocks(s->T);
  if (logits_in == nullptr) {
    TRY(route_from_x(s, x, w_router,
                     route_args(s, nullptr, 1, router_bias, logits_out, topk_idx, topk_gate,
                                partials, err, select_bias),
                     at<float>(ws, L.logits), err, st));
    nb = route_partials_from_x(s);
  } else {
    LAUNCH(launch_route_topk(route_args(s, logits_in, 1, nullptr,
                                        logits_out == logits_in ? nullptr : logits_out, topk_idx,
                                        topk_gate, partials, err, select_bias),
                             st),
           "gates/top-k");
  }
  if (stats) LAUNCH(launch_stats_reduce(partials, nb, s->E, stats, st), "stats reduce");
  return ok();
}

// ---------------------------------------------------------------- backward pass
// Workspace of moe_backward: the forward's layout, then the backward's own buffers.
struct BwdLayout {
  Layout f;
  size_t logits_full, gu, dyp, dO, hbuf, dgu, dxp, dgp, dgate, dl, dl16, dxr, gus, hsb, dgus, dxs;
  size_t total;
};

constexpr int kBwdBn = 256;

BwdLayout layout_bwd(const moe_shape* s) {
  BwdLayout B;
  B.f = layout(s);
  const size_t T = s->T, E = s->E, d = s->d, F = s->d_ff, Fs = s->d_ff_shared;
  const size_t A = perm_rows(s);  // rows: assignments (top-k) or expert-choice rows
  const size_t es = esize(s);
  // dgate partials per row: per column tile and half (bf16), per element (fp32)
  const size_t nt = s->dtype == MOE_BF16 ? 2 * ((F + kBwdBn - 1) / kBwdBn) : F;
  size_t o = B.f.total;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + std::max<size_t>(bytes, 1));
    return at;
  };
  B.logits_full = take(T * E * 4);
  B.gu = take(A * 2 * F * es);
  B.dyp = take(A * d * es);
  B.dO = take(A * d * es);
  B.hbuf = take(A * F * es);
  B.dgu = take(A * 2 * F * es);
  B.dxp = take(A * d * es);
  B.dgp = take(A * nt * 4);
  B.dgate = take(A * 4);
  B.dl = take(T * E * 4);
  B.dl16 = take(T * E * 2);
  B.dxr = take(T * d * es);
  B.gus = take(T * 2 * Fs * es);
  B.hsb = take(T * Fs * es);
  B.dgus = take(T * 2 * Fs * es);
  B.dxs = take(Fs > 0 ? T * d * es : 0);
  B.total = o;
  return B;
}

int check_backward_shape(const moe_shape* s) {
  TRY(check_shape(s));
  if (s->dtype == MOE_F32) return MOE_OK;   // CUDA-core kernels: no tile constraints
  if (s->d % 64 != 0 || s->d_ff % 64 != 0 || s->d_ff_shared % 64 != 0)
    return fail(MOE_ERR_UNSUPPORTED, "the backward pass needs d, d_ff, d_ff_shared multiples of 64");
  if (s->E % 8 != 0) return fail(MOE_ERR_UNSUPPORTED, "the backward pass needs E a multiple of 8");
  return MOE_OK;
}

// One backward GEMM launch; `row_tiles` bounds the DGRAD row tiles (sizes the grid); `mt`
// 256-row weight-gradient tiles (2) or 128-row ones (1).
int bwd_gemm(int mode, BwdProblem p, long long row_tiles, cudaStream_t st, const char* what,
             int mt = 1) {
  const int nt = (p.args.N + kBwdBn - 1) / kBwdBn;
  if (mode == BW_WGRAD)
    p.max_tiles = static_cast<long long>(p.args.groups) * ((p.args.M + 128 * mt - 1) / (128 * mt)) * nt;
  else
    p.max_tiles = row_tiles * nt;
  p.num_sms = num_sms();
  LAUNCH(launch_bwd_gemm(mode, kBwdBn, mt, p, st), what);
  return MOE_OK;
}

int backward_impl(const moe_shape* s, const void* x, const void* w_router, const float* router_bias,
                  const void* w1, const void* w3, const void* w2, const void* w1s, const void* w3s,
                  const void* w2s, const void* dy, float d_aux, float d_z, void* dx, float* dw_router,
                  float* d_router_bias, float* dw1, float* dw3, float* dw2, float* dw1s,
                  float* dw3s, float* dw2s, float* dlogits_out, float* dgate_out, void* ws,
                  size_t ws_bytes, void* stream, void* const* ev, int n_ev) {
  TRY(check_backward_shape(s));
  if (ws == nullptr) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0)
    return fail(MOE_ERR_WORKSPACE, "workspace is not %zu-byte aligned", kAlign);
  const BwdLayout B = layout_bwd(s);
  if (ws_bytes < B.total)
    return fail(MOE_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, B.total);
  if (ev != nullptr && n_ev != MOE_NUM_BWD_STAGES + 1)
    return fail(MOE_ERR_INVALID, "n_events = %d, expected %d", n_ev, MOE_NUM_BWD_STAGES + 1);
  const bool shared = s->d_ff_shared > 0;
  REQUIRE_PTR(dw_router, "dw_router");
  REQUIRE_PTR(dw1, "dw1");
  REQUIRE_PTR(dw3, "dw3");
  REQUIRE_PTR(dw2, "dw2");
  if (shared) {
    REQUIRE_PTR(dw1s, "dw1s");
    REQUIRE_PTR(dw3s, "dw3s");
    REQUIRE_PTR(dw2s, "dw2s");
  }
  OPT_PTR4(router_bias, "router_bias");
  OPT_PTR4(d_router_bias, "d_router_bias");
  OPT_PTR4(dlogits_out, "dlogits_out");
  OPT_PTR4(dgate_out, "dgate_out");
  if (s->T > 0) {
    REQUIRE_PTR(x, "x");
    REQUIRE_PTR(w_router, "w_router");
    REQUIRE_PTR(w1, "w1");
    REQUIRE_PTR(w3, "w3");
    REQUIRE_PTR(w2, "w2");
    REQUIRE_PTR(dy, "dy");
    REQUIRE_PTR(dx, "dx");
    if (shared) {
      REQUIRE_PTR(w1s, "w1s");
      REQUIRE_PTR(w3s, "w3s");
      REQUIRE_PTR(w2s, "w2s");
    }
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto rec = [&](int i) {
    if (ev && ev[i]) cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), st);
  };
  const size_t T = s->T, E = s->E, d = s->d, F = s->d_ff, Fs = s->d_ff_shared;
  const bool ec = expert_choice(s);
  // rows of the permuted activations: T*k assignments, or E*min(C, T) expert-choice rows
  // (whose gate is indexed by the row: perm holds tokens, inv is the dense [T, E] map)
  const size_t A = perm_rows(s);
  const int gather_k = ec ? 1 : s->k;
  const int combine_k = ec ? s->E : s->k;
  const int32_t* gate_perm = nullptr;
  if (s->T == 0) {
    // no tokens: every gradient is 0
    auto zero = [&](void* p, size_t bytes) {
      return p == nullptr || bytes == 0 || cudaMemsetAsync(p, 0, bytes, st) == cudaSuccess;
    };
    if (!zero(dw_router, E * d * 4) || !zero(d_router_bias, E * 4) || !zero(dw1, E * F * d * 4) ||
        !zero(dw3, E * F * d * 4) || !zero(dw2, E * d * F * 4) || !zero(dw1s, Fs * d * 4) ||
        !zero(dw3s, Fs * d * 4) || !zero(dw2s, d * Fs * 4))
      return cuda_status("memset gradients");
    for (int i = 0; ev != nullptr && i < n_ev; ++i) rec(i);
    return ok();
  }
  const Layout& L = B.f;
  DeviceError* err = at<DeviceError>(ws, L.err);
  float* logits = at<float>(ws, B.logits_full);
  int32_t* idx = at<int32_t>(ws, L.idx);
  float* gate = at<float>(ws, L.gate);
  int32_t* cnt = at<int32_t>(ws, L.counts);
  int32_t* off = at<int32_t>(ws, L.offsets);
  int32_t* perm = at<int32_t>(ws, L.perm);
  int32_t* inv = at<int32_t>(ws, L.inv);
  void* xp = at<void>(ws, L.xp);
  void* gu = at<void>(ws, B.gu);
  void* dyp = at<void>(ws, B.dyp);
  void* dO = at<void>(ws, B.dO);
  void* hbuf = at<void>(ws, B.hbuf);
  void* dgu = at<void>(ws, B.dgu);
  void* dxp = at<void>(ws, B.dxp);
  float* dgp = at<float>(ws, B.dgp);
  float* dgate = dgate_out ? dgate_out : at<float>(ws, B.dgate);
  float* dl = dlogits_out ? dlogits_out : at<float>(ws, B.dl);
  void* dl16 = at<void>(ws, B.dl16);
  void* dxr = at<void>(ws, B.dxr);
  void* gus = at<void>(ws, B.gus);
  void* hsb = at<void>(ws, B.hsb);
  void* dgus = at<void>(ws, B.dgus);
  void* dxs = shared ? at<void>(ws, B.dxs) : nullptr;
  const int sms = num_sms();
  const int nt = static_cast<int>(2 * ((F + kBwdBn - 1) / kBwdBn));  // dgate partials per row
  const long long row_tiles = static_cast<long long>((A + 127) / 128) + static_cast<long long>(E);
  const long long row_tiles_T = static_cast<long long>((T + 127) / 128);

  // 1. recompute the routing: logits (with bias), top-k, gates, dispatch -- or the experts'
  //    choices and their gates
  rec(0);
  {
    RouteArgs ra = route_args(s, nullptr, 1, router_bias, logits, idx, gate,
                              at<float>(ws, L.partials), err);
    if (ec) {
      ra.k = 0;  // logits and probabilities only
      ra.probs_t = at<float>(ws, L.probs);
    }
    TRY(route_from_x(s, x, w_router, ra, at<float>(ws, L.logits), err, st));
  }
  if (ec) {
    LAUNCH(launch_expert_choice(at<float>(ws, L.probs), s->T, s->E, s->capacity, perm, gate, inv,
                                cnt, off, at<int32_t>(ws, L.dropped), st),
           "expert choice");
  } else {
    gate_perm = perm;
    LAUNCH(launch_dispatch(idx, s->T * s->k, s->E, s->capacity, cnt, off, perm, inv,
                           at<int32_t>(ws, L.dropped), at<int32_t>(ws, L.blk_hist), err, sms, st),
           "dispatch");
  }
  // inputs of the logit gradient: top-k indices with per-assignment gate gradients, or the
  // dense pair-to-row map with per-row ones; the balance loss is constant under expert choice
  const int32_t* dl_sel = ec ? inv : idx;
  const float dl_aux = ec ? 0.0f : d_aux;
  // 2. gather the rows of x and of dy
  rec(1);
  LAUNCH(launch_gather(x, perm, off, s->E, gather_k, static_cast<int>(d * esize(s)),
                       static_cast<int>(A), xp, sms, st),
         "gather x");
  if (s->dtype == MOE_F32) {
    // fp32 layers: the same steps on the CUDA cores (backward_f32.cu)
    auto f = [](const void* p) { return static_cast<const float*>(p); };
    auto fw = [](void* p) { return static_cast<float*>(p); };
    const int Ai = static_cast<int>(A), Ti = s->T, Ei = s->E, di = s->d, Fi = s->d_ff,
              Fsi = s->d_ff_shared;
    LAUNCH(launch_f32_gather_dy(f(dy), perm, off, gate, Ei, gather_k, ec, di, Ai, fw(dyp),
                                fw(dO), st),
           "gather dy (fp32)");
    rec(2);
    LAUNCH(launch_f32_gu(f(xp), off, Ei, 0, Ai, f(w1), f(w3), Fi, di, fw(gu), st),
           "gate/up recompute (fp32)");
    if (shared)
      LAUNCH(launch_f32_gu(f(x), nullptr, 1, Ti, Ti, f(w1s), f(w3s), Fsi, di, fw(gus), st),
             "shared gate/up recompute (fp32)");
    rec(3);
    LAUNCH(launch_f32_dh(f(dyp), off, Ei, 0, Ai, f(w2), Fi, di, f(gu), gate_perm, gate, fw(dgu),
                         fw(hbuf), dgp, st),
           "dH (fp32)");
    if (shared)
      LAUNCH(launch_f32_dh(f(dy), nullptr, 1, Ti, Ti, f(w2s), Fsi, di, f(gus), nullptr, nullptr,
                           fw(dgus), fw(hsb), nullptr, st),
             "shared dH (fp32)");
    rec(4);
    LAUNCH(launch_dgate(dgp, Fi, ec ? nullptr : inv, Ai, dgate, st), "gate gradient");
    LAUNCH(launch_dlogits(logits, dl_sel, dgate, cnt, Ti, Ei, s->k, s->gate, s->alpha, s->beta,
                          dl_aux, d_z, dl, dl16, st),
           "logit gradient");
    if (d_router_bias != nullptr)
      LAUNCH(launch_column_sum(dl, Ti, Ei, d_router_bias, st), "router bias gradient");
    rec(5);
    LAUNCH(launch_f32_dx(f(dgu), off, Ei, 0, Ai, f(w1), f(w3), Fi, di, fw(dxp), st), "dX (fp32)");
    if (shared)
      LAUNCH(launch_f32_dx(f(dgus), nullptr, 1, Ti, Ti, f(w1s), f(w3s), Fsi, di, fw(dxs), st),
             "shared dX (fp32)");
    LAUNCH(launch_f32_rdx(dl, f(w_router), Ti, Ei, di, fw(dxr), st), "router dX (fp32)");
    rec(6);
    LAUNCH(launch_f32_dx_combine(f(dxp), inv, f(dxr), shared ? f(dxs) : nullptr, Ti, combine_k, di,
                                 fw(dx), st),
           "dx combine (fp32)");
    rec(7);
    LAUNCH(launch_f32_wgrad(f(dgu), 2 * Fi, f(xp), di, off, Ei, 0, 2 * Fi, di, Fi, dw1, dw3, st),
           "dW1/dW3 (fp32)");
    LAUNCH(launch_f32_wgrad(f(dO), di, f(hbuf), Fi, off, Ei, 0, di, Fi, di, dw2, nullptr, st),
           "dW2 (fp32)");
    LAUNCH(launch_f32_wgrad(dl, Ei, f(x), di, nullptr, 1, Ti, Ei, di, Ei, dw_router, nullptr, st),
           "router dW (fp32)");
    if (shared) {
      LAUNCH(launch_f32_wgrad(f(dgus), 2 * Fsi, f(x), di, nullptr, 1, Ti, 2 * Fsi, di, Fsi, dw1s,
                              dw3s, st),
             "shared dW1/dW3 (fp32)");
      LAUNCH(launch_f32_wgrad(f(dy), di, f(hsb), Fsi, nullptr, 1, Ti, di, Fsi, di, dw2s, nullptr,
                              st),
             "shared dW2 (fp32)");
    }
    rec(8);
    return ok();
  }
  LAUNCH(launch_gather_dy(dy, perm, off, gate, s->E, gather_k, ec, s->d, static_cast<int>(A), dyp,
                          dO, sms, st),
         "gather dy");
  // 3. recompute the pre-activations G | U (routed experts and the shared expert)
  rec(2);
  {
    TcProblem p{};
    p.args.groups = s->E;
    p.args.offsets = off;
    p.args.n_routed = s->d_ff;
    p.args.k_routed = s->d;
    p.args.out_routed = nullptr;
    p.args.gu_routed = gu;
    p.args.has_shared = shared;
    p.args.m_shared = s->T;
    p.args.n_shared = s->d_ff_shared;
    p.args.k_shared = s->d;
    p.args.out_shared = nullptr;
    p.args.gu_shared = gus;
    p.args.err = err;
    p.a = xp;
    p.a_rows = static_cast<long long>(A);
    p.b0 = w1;
    p.b1 = w3;
    p.b_rows = s->d_ff;
    p.b_groups = s->E;
    p.a_s = x;
    p.b0_s = w1s;
    p.b1_s = w3s;
    p.b_rows_s = s->d_ff_shared;
    // the forward's row-tile policy: 256-row tiles when experts average >= 512 rows
    const int mt_gu = (A / s->E >= 512 && s->E <= kTcMt2MaxGroups) ? 2 : 1;
    const long long tm = 128ll * mt_gu;
    p.max_tiles = (static_cast<long long>((A + tm - 1) / tm) + static_cast<long long>(E)) *
                      ((s->d_ff + 127) / 128) +
                  (shared ? static_cast<long long>((T + tm - 1) / tm) * ((s->d_ff_shared + 127) / 128)
                          : 0);
    p.num_sms = sms;
    LAUNCH(launch_tc_gemm(TC_SWIGLU, 256, mt_gu, 64, false, 128, p, st),
           "gate/up recompute (tcgen05)");
  }
  // 4. dH_raw = dy W2 with the SwiGLU backward and the gate-gradient partials
  rec(3);
  {
    BwdProblem p{};
    p.args.groups = s->E;
    p.args.offsets = off;
    p.args.N = s->d_ff;
    p.args.K = s->d;
    p.args.gu = gu;
    p.args.dgu = dgu;
    p.args.h = hbuf;
    p.args.dg_part = dgp;
    p.args.n_tiles = nt;
    p.args.perm = gate_perm;
    p.args.gate = gate;
    p.args.err = err;
    p.a = dyp;
    p.a_rows = static_cast<long long>(A);
    p.b0 = w2;
    p.b_inner = s->d_ff;
    p.b_rows = s->d;
    p.b_groups = s->E;
    TRY(bwd_gemm(BW_DGRAD_H, p, row_tiles, st, "dH GEMM (tcgen05)"));
    if (shared) {
      BwdProblem q{};
      q.args.groups = 1;
      q.args.m_single = s->T;
      q.args.N = s->d_ff_shared;
      q.args.K = s->d;
      q.args.gu = gus;
      q.args.dgu = dgus;
      q.args.h = hsb;
      q.args.err = err;
      q.a = dy;
      q.a_rows = s->T;
      q.b0 = w2s;
      q.b_inner = s->d_ff_shared;
      q.b_rows = s->d;
      q.b_groups = 1;
      TRY(bwd_gemm(BW_DGRAD_H, q, row_tiles_T, st, "shared dH GEMM (tcgen05)"));
    }
  }
  // 5. gate gradients -> router logit gradients (gates, balance loss, z-loss)
  rec(4);
  LAUNCH(launch_dgate(dgp, nt, ec ? nullptr : inv, static_cast<int>(A), dgate, st), "gate gradient");
  LAUNCH(launch_dlogits(logits, dl_sel, dgate, cnt, s->T, s->E, s->k, s->gate, s->alpha, s->beta,
                        dl_aux, d_z, dl, dl16, st),
         "logit gradient");
  if (d_router_bias != nullptr)
    LAUNCH(launch_column_sum(dl, s->T, s->E, d_router_bias, st), "router bias gradient");
  // 6. dXp = dG W1 + dU W3 (routed, shared) and the router's dx = dl W_r
  rec(5);
  {
    BwdProblem p{};
    p.args.groups = s->E;
    p.args.offsets = off;
    p.args.N = s->d;
    p.args.K = 2 * s->d_ff;
    p.args.k_split = s->d_ff;
    p.args.out = dxp;
    p.args.ldo = s->d;
    p.args.err = err;
    p.a = dgu;
    p.a_rows = static_cast<long long>(A);
    p.b0 = w1;
    p.b1 = w3;
    p.b_inner = s->d;
    p.b_rows = s->d_ff;
    p.b_groups = s->E;
    TRY(bwd_gemm(BW_DGRAD_X, p, row_tiles, st, "dX GEMM (tcgen05)"));
    if (shared) {
      BwdProblem q = p;
      q.args.groups = 1;
      q.args.offsets = nullptr;
      q.args.m_single = s->T;
      q.args.K = 2 * s->d_ff_shared;
      q.args.k_split = s->d_ff_shared;
      q.args.out = dxs;
      q.a = dgus;
      q.a_rows = s->T;
      q.b0 = w1s;
      q.b1 = w3s;
      q.b_rows = s->d_ff_shared;
      q.b_groups = 1;
      TRY(bwd_gemm(BW_DGRAD_X, q, row_tiles_T, st, "shared dX GEMM (tcgen05)"));
    }
    BwdProblem r{};
    r.args.groups = 1;
    r.args.m_single = s->T;
    r.args.N = s->d;
    r.args.K = s->E;
    r.args.k_split = s->E;
    r.args.out = dxr;
    r.args.ldo = s->d;
    r.args.err = err;
    r.a = dl16;
    r.a_rows = s->T;
    r.b0 = w_router;
    r.b_inner = s->d;
    r.b_rows = s->E;
    r.b_groups = 1;
    TRY(bwd_gemm(BW_DGRAD_X, r, row_tiles_T, st, "router dX GEMM (tcgen05)"));
  }
  rec(6);
  LAUNCH(launch_dx_combine(dxp, inv, dxr, dxs, dx, s->T, combine_k, s->d, sms, st), "dx combine");
  // 7. weight gradients: per expert dW1 | dW3 = [dG dU]^T Xp, dW2 = (g dy)^T H; router; shared
  rec(7);
  {
    BwdProblem p{};
    p.args.groups = s->E;
    p.args.offsets = off;
    p.args.M = 2 * s->d_ff;
    p.args.m_split = s->d_ff;
    p.args.N = s->d;
    p.args.out = dw1;
    p.args.out1 = dw3;
    p.args.err = err;
    p.a = dgu;
    p.a_rows = static_cast<long long>(A);
    p.a_inner = 2 * s->d_ff;
    p.b0 = xp;
    p.b_rows = static_cast<long long>(A);
    p.b_inner = s->d;
    // Experts with many rows (long K per output tile): 256-row tiles, twice the MMA work per
    // staged byte (the weight-gradient GEMMs read both operands through L2); few rows: 128.
    const int mt_w = (A / s->E >= 512) ? 2 : 1;
    TRY(bwd_gemm(BW_WGRAD, p, 0, st, "dW1/dW3 GEMM (tcgen05)", mt_w));
    BwdProblem q = p;
    q.args.M = s->d;
    q.args.m_split = s->d;
    q.args.N = s->d_ff;
    q.args.out = dw2;
    q.args.out1 = nullptr;
    q.a = dO;
    q.a_inner = s->d;
    q.b0 = hbuf;
    q.b_inner = s->d_ff;
    TRY(bwd_gemm(BW_WGRAD, q, 0, st, "dW2 GEMM (tcgen05)", mt_w));
    BwdProblem r{};
    r.args.groups = 1;
    r.args.m_single = s->T;
    r.args.M = s->E;
    r.args.m_split = s->E;
    r.args.N = s->d;
    r.args.out = dw_router;
    r.args.err = err;
    r.a = dl16;
    r.a_rows = s->T;
    r.a_inner = s->E;
    r.b0 = x;
    r.b_rows = s->T;
    r.b_inner = s->d;
    TRY(bwd_gemm(BW_WGRAD, r, 0, st, "router dW GEMM (tcgen05)"));
    if (shared) {
      BwdProblem u = r;
      u.args.M = 2 * s->d_ff_shared;
      u.args.m_split = s->d_ff_shared;
      u.args.out = dw1s;
      u.args.out1 = dw3s;
      u.a = dgus;
      u.a_inner = 2 * s->d_ff_shared;
      TRY(bwd_gemm(BW_WGRAD, u, 0, st, "shared dW1/dW3 GEMM (tcgen05)"));
      BwdProblem v = r;
      v.args.M = s->d;
      v.args.m_split = s->d;
      v.args.N = s->d_ff_shared;
      v.args.out = dw2s;
      v.a = dy;
      v.a_inner = s->d;
      v.b0 = hsb;
      v.b_inner = s->d_ff_shared;
      TRY(bwd_gemm(BW_WGRAD, v, 0, st, "shared dW2 GEMM (tcgen05)"));
    }
  }
  rec(8);
  return ok();
}
}  // namespace

extern "C" {

int moe_route_topk(const moe_shape* s, const void* x, const void* w_router,
                   const float* router_bias, const float* logits_in, float* logits_out,
                   int32_t* topk_idx, float* topk_gate, float* stats, void* ws, size_t ws_bytes,
                   void* stream) {
  return route_impl(s, x, w_router, router_bias, logits_in, nullptr, logits_out, topk_idx,
                    topk_gate, stats, ws, ws_bytes, stream);
}

int moe_route_topk_balanced(const moe_shape* s, const void* x, const void* w_router,
                            const float* router_bias, const float* logits_in,
                            const float* select_bias, float* logits_out, int32_t* topk_idx,
                            float* topk_gate, float* stats, void* ws, size_t ws_bytes,
                            void* stream) {
  if (select_bias == nullptr) return fail(MOE_ERR_INVALID, "select_bias is NULL");
  if (!aligned4(select_bias)) return fail(MOE_ERR_INVALID, "select_bias is not 4-byte aligned");
  return route_impl(s, x, w_router, router_bias, logits_in, select_bias, logits_out, topk_idx,
                    topk_gate, stats, ws, ws_bytes, stream);
}

int moe_expert_choice(const moe_shape* s, const void* x, const void* w_router,
                      const float* router_bias, const float* logits_in, int32_t* perm,
                      int32_t* offsets, float* row_gate, int32_t* inv, int32_t* counts,
                      int32_t* unrouted, float* stats, void* ws, size_t ws_bytes, void* stream) {
  TRY(check_shape(s));
  if (!expert_choice(s))
    return fail(MOE_ERR_INVALID, "moe_expert_choice needs gate = MOE_GATE_EXPERT_CHOICE");
  TRY(check_ws(s, ws, ws_bytes));
  REQUIRE_PTR4(offsets, "offsets");
  REQUIRE_PTR4(counts, "counts");
  REQUIRE_PTR4(unrouted, "unrouted");
  OPT_PTR4(stats, "stats");
  if (s->T > 0) {
    if (logits_in == nullptr) {
      REQUIRE_PTR(x, "x");
      REQUIRE_PTR(w_router, "w_router");
      OPT_PTR4(router_bias, "router_bias");
    } else {
      REQUIRE_PTR4(logits_in, "logits_in");
    }
    REQUIRE_PTR4(perm, "perm");
    REQUIRE_PTR4(row_gate, "row_gate");
    REQUIRE_PTR4(inv, "inv");
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Layout L = layout(s);
  DeviceError* err = at<DeviceError>(ws, L.err);
  float* partials = at<float>(ws, L.partials);
  if (s->T > 0) {
    int nb = route_blocks(s->T);
    if (logits_in == nullptr) {
      RouteArgs ra = route_args(s, nullptr, 1, router_bias, nullptr, nullptr, nullptr, partials,
                                err);
      ra.k = 0;
      ra.probs_t = at<float>(ws, L.probs);
      TRY(route_from_x(s, x, w_router, ra, at<float>(ws, L.logits), err, st));
      nb = route_partials_from_x(s);
    } else {
      RouteArgs ra = route_args(s, logits_in, 1, nullptr, nullptr, nullptr, nullptr, partials,
                                err);
      ra.k = 0;
      ra.probs_t = at<float>(ws, L.probs);
      LAUNCH(launch_route_topk(ra, st), "router probabilities");
    }
    if (stats) LAUNCH(launch_stats_reduce(partials, nb, s->E, stats, st), "stats reduce");
  } else if (stats && cudaMemsetAsync(stats, 0, (s->E + 1) * sizeof(float), st) != cudaSuccess) {
    return cuda_status("memset stats");
  }
  LAUNCH(launch_expert_choice(at<float>(ws, L.probs), s->T, s->E, s->capacity, perm, row_gate,
                              inv, counts, offsets, unrouted, st),
         "expert choice");
  return ok();
}

int moe_grouped_swiglu_fp8w(const moe_shape* s, const void* x, const int32_t* perm,
                            const int32_t* offsets, const float* topk_gate, const uint8_t* w1q,
                            const float* w1_scale, const uint8_t* w3q, const float* w3_scale,
                            const uint8_t* w2q, const float* w2_scale, void* y_perm, void* ws,
                            size_t ws_bytes, void* stream) {
  TRY(check_shape(s));
  TRY(check_ws(s, ws, ws_bytes));
  const Fp8Weights q{w1q, w3q, w2q, w1_scale, w3_scale, w2_scale};
  TRY(check_fp8(s, &q));
  if (s->T == 0) return ok();
  REQUIRE_PTR(x, "x");
  REQUIRE_PTR4(perm, "perm");
  REQUIRE_PTR4(offsets, "offsets");
  OPT_PTR4(topk_gate, "topk_gate");
  REQUIRE_PTR(y_perm, "y_perm");
  const bool ec = expert_choice(s);
  TRY(run_experts(s, x, perm, offsets, ec ? nullptr : topk_gate, ec ? topk_gate : nullptr, nullptr,
                  nullptr, nullptr, nullptr, nullptr, nullptr, y_perm, nullptr, ws,
                  static_cast<cudaStream_t>(stream), nullptr, 0, &q));
  return ok();
}

int moe_forward_fp8w(const moe_shape* s, const void* x, const void* w_router,
                     const float* router_bias, const uint8_t* w1q, const float* w1_scale,
                     const uint8_t* w3q, const float* w3_scale, const uint8_t* w2q,
                     const float* w2_scale, void* y, int32_t* counts, int32_t* dropped,
                     float* losses, void* ws, size_t ws_bytes, void* stream, void* const* events,
                     int n_events) {
  const Fp8Weights q{w1q, w3q, w2q, w1_scale, w3_scale, w2_scale};
  return forward_impl(s, x, w_router, router_bias, nullptr, nullptr, nullptr, nullptr, nullptr,
                      nullptr, y, counts, dropped, losses, ws, ws_bytes, stream, events,
                      events ? n_events : 0, nullptr, 0.f, &q);
}

int moe_update_select_bias(const moe_shape* s, const int32_t* counts, float* select_bias,
                           float gamma, void* stream) {
  TRY(check_shape(s));
  REQUIRE_PTR4(counts, "counts");
  REQUIRE_PTR4(select_bias, "select_bias");
  if (!(gamma >= 0.f)) return fail(MOE_ERR_INVALID, "gamma must be >= 0");
  LAUNCH(launch_update_select_bias(counts, select_bias, s->T, s->E, s->k, gamma,
                                   static_cast<cudaStream_t>(stream)),
         "selection bias update");
  return ok();
}

int moe_forward_balanced(const moe_shape* s, const void* x, const void* w_router,
                         const float* router_bias, const void* w1, const void* w3, const void* w2,
                         const void* w1s, const void* w3s, const void* w2s, void* y,
                         int32_t* counts, int32_t* dropped, float* losses, float* select_bias,
                         float gamma, void* ws, size_t ws_bytes, void* stream,
                         void* const* events, int n_events) {
  if (select_bias == nullptr) return fail(MOE_ERR_INVALID, "select_bias is NULL");
  if (!aligned4(select_bias)) return fail(MOE_ERR_INVALID, "select_bias is not 4-byte aligned");
  if (!(gamma >= 0.f)) return fail(MOE_ERR_INVALID, "gamma must be >= 0");
  return forward_impl(s, x, w_router, router_bias, w1, w3, w2, w1s, w3s, w2s, y, counts, dropped,
                      losses, ws, ws_bytes, stream, events, events ? n_events : 0, select_bias,
                      gamma);
}

int moe_dispatch(const moe_shape* s, const int32_t* topk_idx, const float* logits_in,
                 int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* dropped,
                 void* ws, size_t ws_bytes, void* stream) {
  TRY(check_shape(s));
  if (expert_choice(s))
    return fail(MOE_ERR_UNSUPPORTED, "expert-choice layers route with moe_expert_choice");
  TRY(check_ws(s, ws, ws_bytes));
  REQUIRE_PTR4(counts, "counts");
  REQUIRE_PTR4(offsets, "offsets");
  REQUIRE_PTR4(dropped, "dropped");
  if (s->T > 0) {
    if (topk_idx == nullptr) REQUIRE_PTR4(logits_in, "logits_in (topk_idx is NULL)");
    else REQUIRE_PTR4(topk_idx, "topk_idx");
    REQUIRE_PTR4(perm, "perm");
    REQUIRE_PTR4(inv, "inv");
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Layout L = layout(s);
  DeviceError* err = at<DeviceError>(ws, L.err);
  const int32_t* idx = topk_idx;
  if (idx == nullptr && s->T > 0) {
    int32_t* widx = at<int32_t>(ws, L.idx);
    LAUNCH(launch_route_topk(route_args(s, logits_in, 1, nullptr, nullptr, widx,
                                        at<float>(ws, L.gate), at<float>(ws, L.partials), err),
                             st),
           "gates/top-k");
    idx = widx;
  }
  LAUNCH(launch_dispatch(idx, s->T * s->k, s->E, s->capacity, counts, offsets, perm, inv, dropped,
                         at<int32_t>(ws, L.blk_hist), err, num_sms(), st),
         "dispatch");
  return ok();
}

int moe_grouped_swiglu(const moe_shape* s, const void* x, const int32_t* perm,
                       const int32_t* offsets, const float* topk_gate, const void* w1,
                       const void* w3, const void* w2, const void* w1s, const void* w3s,
                       const void* w2s, void* y_perm, void* y_shared, void* ws, size_t ws_bytes,
                       void* stream) {
  TRY(check_shape(s));
  TRY(check_ws(s, ws, ws_bytes));
  if (s->T == 0) return ok();
  REQUIRE_PTR(x, "x");
  REQUIRE_PTR4(perm, "perm");
  REQUIRE_PTR4(offsets, "offsets");
  OPT_PTR4(topk_gate, "topk_gate");
  REQUIRE_PTR(w1, "w1");
  REQUIRE_PTR(w3, "w3");
  REQUIRE_PTR(w2, "w2");
  REQUIRE_PTR(y_perm, "y_perm");
  if (s->d_ff_shared > 0) {
    REQUIRE_PTR(w1s, "w1s");
    REQUIRE_PTR(w3s, "w3s");
    REQUIRE_PTR(w2s, "w2s");
    REQUIRE_PTR(y_shared, "y_shared");
  }
  const bool ec = expert_choice(s);
  TRY(run_experts(s, x, perm, offsets, ec ? nullptr : topk_gate, ec ? topk_gate : nullptr, w1, w3,
                  w2, w1s, w3s, w2s, y_perm, s->d_ff_shared > 0 ? y_shared : nullptr, ws,
                  static_cast<cudaStream_t>(stream), nullptr, 0));
  return ok();
}

int moe_combine(const moe_shape* s, const void* y_perm, const int32_t* inv, const void* y_shared,
                void* y, void* stream) {
  TRY(check_shape(s));
  if (s->T == 0) return ok();
  REQUIRE_PTR(y_perm, "y_perm");
  REQUIRE_PTR4(inv, "inv");
  REQUIRE_PTR(y, "y");
  if (y_shared != nullptr && !aligned16(y_shared))
    return fail(MOE_ERR_INVALID, "y_shared is not 16-byte aligned");
  LAUNCH(launch_combine(s->dtype, y_perm, inv, y_shared, y, s->T,
                        expert_choice(s) ? s->E : s->k, s->d, num_sms(),
                        static_cast<cudaStream_t>(stream)),
         "combine");
  return ok();
}

int moe_aux_loss(const moe_shape* s, const float* stats, const int32_t* counts, float* losses,
                 void* stream) {
  TRY(check_shape(s));
  REQUIRE_PTR4(stats, "stats");
  REQUIRE_PTR4(counts, "counts");
  REQUIRE_PTR4(losses, "losses");
  LAUNCH(launch_aux_loss(stats, counts, s->T, s->E, s->k, s->alpha, s->beta, losses,
                         static_cast<cudaStream_t>(stream)),
         "aux loss");
  return ok();
}

int moe_forward(const moe_shape* s, const void* x, const void* w_router, const float* router_bias,
                const void* w1, const void* w3, const void* w2, const void* w1s, const void* w3s,
                const void* w2s, void* y, int32_t* counts, int32_t* dropped, float* losses,
                void* ws, size_t ws_bytes, void* stream) {
  return forward_impl(s, x, w_router, router_bias, w1, w3, w2, w1s, w3s, w2s, y, counts, dropped,
                      losses, ws, ws_bytes, stream, nullptr, 0);
}

int moe_forward_host(const moe_shape* s, const void* x_host, const void* w_router,
                     const float* router_bias, const void* w1, const void* w3, const void* w2,
                     const void* w1s, const void* w3s, const void* w2s, void* y_host,
                     float* losses_host, void* x_dev, void* y_dev, void* ws, size_t ws_bytes,
                     void* stream) {
  TRY(check_forward(s, x_dev, w_router, router_bias, w1, w3, w2, w1s, w3s, w2s, y_dev, nullptr,
                    nullptr, nullptr, ws, ws_bytes, nullptr, 0, nullptr));
  const size_t bytes = static_cast<size_t>(s->T) * s->d * esize(s);
  if (s->T > 0) {
    if (x_host == nullptr) return fail(MOE_ERR_INVALID, "x_host is NULL");
    if (y_host == nullptr) return fail(MOE_ERR_INVALID, "y_host is NULL");
  }
  OPT_PTR4(losses_host, "losses_host");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (bytes > 0 && cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return cuda_status("copy x to the device");
  TRY(forward_impl(s, x_dev, w_router, router_bias, w1, w3, w2, w1s, w3s, w2s, y_dev, nullptr,
                   nullptr, nullptr, ws, ws_bytes, stream, nullptr, 0));
  if (bytes > 0 && cudaMemcpyAsync(y_host, y_dev, bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return cuda_status("copy y to the host");
  if (losses_host != nullptr &&
      cudaMemcpyAsync(losses_host, at<float>(ws, layout(s).losses), 2 * sizeof(float),
                      cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return cuda_status("copy the losses to the host");
  return ok();
}

#define CUDA_TRY(expr, what)                                                          \
  do {                                                                                \
    const cudaError_t e_ = (expr);                                                    \
    if (e_ != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e_)); \
  } while (0)

struct moe_host_pipeline {
  int d = 0, dtype = 0;
  int64_t max_T = 0;
  cudaStream_t up = nullptr, down = nullptr;
  void* x_dev[2] = {nullptr, nullptr};
  void* y_dev[2] = {nullptr, nullptr};
  float* losses_dev[2] = {nullptr, nullptr};
  // per slot: its upload finished / its layer finished / its download finished
  cudaEvent_t uploaded[2] = {nullptr, nullptr};
  cudaEvent_t layer_done[2] = {nullptr, nullptr};
  cudaEvent_t downloaded[2] = {nullptr, nullptr};
  uint64_t step = 0;
};

int moe_host_pipeline_destroy(moe_host_pipeline* p) {
  if (p == nullptr) return MOE_OK;
  int rc = MOE_OK;
  auto note = [&](cudaError_t e, const char* what) {
    if (e != cudaSuccess && rc == MOE_OK) rc = fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  };
  // the buffers may still be read by queued copies or layers
  for (int b = 0; b < 2; ++b)
    if (p->layer_done[b]) note(cudaEventSynchronize(p->layer_done[b]), "wait for a layer");
  if (p->up) note(cudaStreamSynchronize(p->up), "wait for the uploads");
  if (p->down) note(cudaStreamSynchronize(p->down), "wait for the downloads");
  for (int b = 0; b < 2; ++b) {
    for (cudaEvent_t e : {p->uploaded[b], p->layer_done[b], p->downloaded[b]})
      if (e) note(cudaEventDestroy(e), "destroy an event");
  }
  if (p->up) note(cudaStreamDestroy(p->up), "destroy the upload stream");
  if (p->down) note(cudaStreamDestroy(p->down), "destroy the download stream");
  delete p;
  return rc;
}

// The caller's buffer, slot by slot: x [T_max, d], y [T_max, d], losses [2], each rounded up
// to kAlign bytes.
size_t pipeline_slot_bytes(const moe_shape* s) {
  const size_t rows = static_cast<size_t>(s->T) * s->d * esize(s);
  const size_t r = (rows + kAlign - 1) / kAlign * kAlign;
  return 2 * r + kAlign;
}

static int pipeline_setup(moe_host_pipeline* p, const moe_shape* s, void* buf) {
  p->d = s->d;
  p->dtype = s->dtype;
  p->max_T = s->T;
  const size_t slot = pipeline_slot_bytes(s);
  const size_t rows = (slot - kAlign) / 2;
  for (int b = 0; b < 2; ++b) {
    uint8_t* base = static_cast<uint8_t*>(buf) + b * slot;
    p->x_dev[b] = base;
    p->y_dev[b] = base + rows;
    p->losses_dev[b] = reinterpret_cast<float*>(base + 2 * rows);
  }
  CUDA_TRY(cudaStreamCreateWithFlags(&p->up, cudaStreamNonBlocking), "create the upload stream");
  CUDA_TRY(cudaStreamCreateWithFlags(&p->down, cudaStreamNonBlocking), "create the download stream");
  for (int b = 0; b < 2; ++b)
    for (cudaEvent_t* e : {&p->uploaded[b], &p->layer_done[b], &p->downloaded[b]})
      CUDA_TRY(cudaEventCreateWithFlags(e, cudaEventDisableTiming), "create an event");
  return MOE_OK;
}

size_t moe_host_pipeline_buffer_size(const moe_shape* s_max) {
  if (check_shape(s_max) != MOE_OK) return 0;
  return 2 * pipeline_slot_bytes(s_max);
}

int moe_host_pipeline_create(const moe_shape* s_max, void* buf, size_t buf_bytes,
                             moe_host_pipeline** out) {
  if (out == nullptr) return fail(MOE_ERR_INVALID, "out is NULL");
  *out = nullptr;
  TRY(check_shape(s_max));
  if (buf == nullptr) return fail(MOE_ERR_WORKSPACE, "pipeline buffer is NULL");
  if ((reinterpret_cast<uintptr_t>(buf) & (kAlign - 1)) != 0)
    return fail(MOE_ERR_WORKSPACE, "pipeline buffer is not %zu-byte aligned", kAlign);
  const size_t need = 2 * pipeline_slot_bytes(s_max);
  if (buf_bytes < need)
    return fail(MOE_ERR_WORKSPACE, "pipeline buffer has %zu bytes, needs %zu", buf_bytes, need);
  auto* p = new moe_host_pipeline();
  const int rc = pipeline_setup(p, s_max, buf);
  if (rc != MOE_OK) {
    moe_host_pipeline_destroy(p);
    return rc;
  }
  *out = p;
  return ok();
}

int moe_host_pipeline_forward(moe_host_pipeline* p, const moe_shape* s, const void* x_host,
                              const void* w_router, const float* router_bias, const void* w1,
                              const void* w3, const void* w2, const void* w1s, const void* w3s,
                              const void* w2s, void* y_host, float* losses_host, void* ws,
                              size_t ws_bytes, void* stream) {
  if (p == nullptr) return fail(MOE_ERR_INVALID, "pipeline is NULL");
  TRY(check_shape(s));
  if (s->d != p->d || s->dtype != p->dtype || s->T > p->max_T)
    return fail(MOE_ERR_INVALID, "shape (T %lld, d %d, dtype %d) outside the pipeline's "
                "(T <= %lld, d %d, dtype %d)", static_cast<long long>(s->T), s->d, s->dtype,
                static_cast<long long>(p->max_T), p->d, p->dtype);
  const int b = static_cast<int>(p->step & 1);
  TRY(check_forward(s, p->x_dev[b], w_router, router_bias, w1, w3, w2, w1s, w3s, w2s,
                    p->y_dev[b], nullptr, nullptr, p->losses_dev[b], ws, ws_bytes, nullptr, 0,
                    nullptr));
  if (s->T > 0) {
    if (x_host == nullptr) return fail(MOE_ERR_INVALID, "x_host is NULL");
    if (y_host == nullptr) return fail(MOE_ERR_INVALID, "y_host is NULL");
  }
  OPT_PTR4(losses_host, "losses_host");
  const size_t bytes = static_cast<size_t>(s->T) * s->d * esize(s);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // upload into the slot once the layer that last read its x is done
  CUDA_TRY(cudaStreamWaitEvent(p->up, p->layer_done[b], 0), "order the upload");
  if (bytes > 0)
    CUDA_TRY(cudaMemcpyAsync(p->x_dev[b], x_host, bytes, cudaMemcpyHostToDevice, p->up),
             "copy x to the device");
  CUDA_TRY(cudaEventRecord(p->uploaded[b], p->up), "record the upload");
  // the layer: after its upload and after the download that last read the slot's outputs
  CUDA_TRY(cudaStreamWaitEvent(st, p->uploaded[b], 0), "order the layer");
  CUDA_TRY(cudaStreamWaitEvent(st, p->downloaded[b], 0), "order the layer");
  TRY(forward_impl(s, p->x_dev[b], w_router, router_bias, w1, w3, w2, w1s, w3s, w2s, p->y_dev[b],
                   nullptr, nullptr, p->losses_dev[b], ws, ws_bytes, stream, nullptr, 0));
  CUDA_TRY(cudaEventRecord(p->layer_done[b], st), "record the layer");
  // download
  CUDA_TRY(cudaStreamWaitEvent(p->down, p->layer_done[b], 0), "order the download");
  if (bytes > 0)
    CUDA_TRY(cudaMemcpyAsync(y_host, p->y_dev[b], bytes, cudaMemcpyDeviceToHost, p->down),
             "copy y to the host");
  if (losses_host != nullptr)
    CUDA_TRY(cudaMemcpyAsync(losses_host, p->losses_dev[b], 2 * sizeof(float),
                             cudaMemcpyDeviceToHost, p->down),
             "copy the losses to the host");
  CUDA_TRY(cudaEventRecord(p->downloaded[b], p->down), "record the download");
  ++p->step;
  return ok();
}

int moe_host_pipeline_join(moe_host_pipeline* p, void* stream) {
  if (p == nullptr) return fail(MOE_ERR_INVALID, "pipeline is NULL");
  for (int b = 0; b < 2; ++b)
    CUDA_TRY(cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), p->downloaded[b], 0),
             "join the downloads");
  return ok();
}

int moe_forward_events(const moe_shape* s, const void* x, const void* w_router,
                       const float* router_bias, const void* w1, const void* w3, const void* w2,
                       const void* w1s, const void* w3s, const void* w2s, void* y,
                       int32_t* counts, int32_t* dropped, float* losses, void* ws,
                       size_t ws_bytes, void* stream, void* const* events, int n_events) {
  if (events == nullptr) return fail(MOE_ERR_INVALID, "events is NULL");
  return forward_impl(s, x, w_router, router_bias, w1, w3, w2, w1s, w3s, w2s, y, counts, dropped,
                      losses, ws, ws_bytes, stream, events, n_events);
}

int moe_get_error(const void* ws, void* stream) {
  if (ws == nullptr) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
  DeviceError h{};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return cuda_status("read error word");
  if (cudaStreamSynchronize(st) != cudaSuccess) return cuda_status("synchronize");
  if (h.code != 0) {
    g_detail = "device error at site " + std::to_string(h.where) + ", detail " +
               std::to_string(h.detail);
    return h.code;
  }
  return ok();
}

int moe_selftest_wait_timeout(void* ws, size_t ws_bytes, void* stream) {
  if (ws == nullptr) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0)
    return fail(MOE_ERR_WORKSPACE, "workspace is not %zu-byte aligned", kAlign);
  if (ws_bytes < sizeof(DeviceError))
    return fail(MOE_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes,
                sizeof(DeviceError));
  LAUNCH(launch_wait_timeout(static_cast<DeviceError*>(ws), static_cast<cudaStream_t>(stream)),
         "bounded-wait self-test");
  return ok();
}

int moe_workspace_dispatch_offsets(const moe_shape* s, size_t* perm_offset, size_t* inv_offset,
                                   size_t* offsets_offset) {
  TRY(check_shape(s));
  if (perm_offset == nullptr || inv_offset == nullptr || offsets_offset == nullptr)
    return fail(MOE_ERR_INVALID, "an output pointer is NULL");
  if (expert_choice(s))
    return fail(MOE_ERR_UNSUPPORTED, "expert-choice layers keep token rows, not a dispatch");
  const Layout L = layout(s);
  *perm_offset = L.perm;
  *inv_offset = L.inv;
  *offsets_offset = L.offsets;
  return ok();
}

int moe_clear_error(void* ws, void* stream) {
  if (ws == nullptr) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
  if (cudaMemsetAsync(ws, 0, sizeof(DeviceError), static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return cuda_status("clear error word");
  return ok();
}

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_NONFINITE: return "non-finite value (router logit, or beyond fp16 on the 8-bit path)";
    default: return "unknown status";
  }
}

const char* moe_last_error_detail(void) { return g_detail.c_str(); }

size_t moe_backward_workspace_size(const moe_shape* s) {
  if (check_backward_shape(s) != MOE_OK) return 0;
  return layout_bwd(s).total;
}

int moe_backward(const moe_shape* s, const void* x, const void* w_router, const float* router_bias,
                 const void* w1, const void* w3, const void* w2, const void* w1s, const void* w3s,
                 const void* w2s, const void* dy, float d_aux, float d_z, void* dx,
                 float* dw_router, float* d_router_bias, float* dw1, float* dw3, float* dw2,
                 float* dw1s, float* dw3s, float* dw2s, float* dlogits, float* dgate, void* ws,
                 size_t ws_bytes, void* stream, void* const* events, int n_events) {
  return backward_impl(s, x, w_router, router_bias, w1, w3, w2, w1s, w3s, w2s, dy, d_aux, d_z, dx,
                       dw_router, d_router_bias, dw1, dw3, dw2, dw1s, dw3s, dw2s, dlogits, dgate,
                       ws, ws_bytes, stream, events, n_events);
}


size_t moe_mx_workspace_size(const moe_shape* s) {
  if (check_shape(s) != MOE_OK) return 0;
  return layout_mx(s).total;
}

int moe_forward_mx(const moe_shape* s, int fmt, const void* x, const void* w_router,
                   const float* router_bias, const uint8_t* w1q, const uint8_t* w1_scales,
                   const uint8_t* w3q, const uint8_t* w3_scales, const uint8_t* w2q,
                   const uint8_t* w2_scales, void* y, int32_t* counts, int32_t* dropped,
                   float* losses, void* ws, size_t ws_bytes, void* stream, void* const* events,
                   int n_events) {
  const MxWeights m{fmt, w1q, w3q, w2q, w1_scales, w3_scales, w2_scales};
  return forward_impl(s, x, w_router, router_bias, nullptr, nullptr, nullptr, nullptr, nullptr,
                      nullptr, y, counts, dropped, losses, ws, ws_bytes, stream, events,
                      events ? n_events : 0, nullptr, 0.f, nullptr, &m);
}

int moe_mx_quantize(const void* x, int64_t rows, int32_t K, uint8_t* codes, uint8_t* scales,
                    void* ws, void* stream) {
  if (rows < 0) return fail(MOE_ERR_INVALID, "rows = %lld < 0", static_cast<long long>(rows));
  if (K < 32 || K % 32 != 0) return fail(MOE_ERR_INVALID, "K = %d is not a positive multiple of 32", K);
  if (rows > 0) {
    REQUIRE_PTR(x, "x");
    REQUIRE_PTR(codes, "codes");
    if (scales == nullptr) return fail(MOE_ERR_INVALID, "scales is NULL");
  }
  if (ws != nullptr && (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0)
    return fail(MOE_ERR_WORKSPACE, "workspace is not %zu-byte aligned", kAlign);
  LAUNCH(launch_mx_quant_rows(x, rows, K, codes, scales, static_cast<DeviceError*>(ws),
                              static_cast<cudaStream_t>(stream)),
         "block quantization");
  return ok();
}
}  // extern "C"
