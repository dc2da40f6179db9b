// Grouped GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// One persistent kernel computes C = A . B^T for a list of groups that share B's shape:
// the routed experts (group e owns the contiguous rows [offsets[e], offsets[e+1]) of A and
// the weight slice B[e]) and, optionally, one always-active shared expert (rows [0, M_s)
// of its own A and B). This is the "grouped GEMM over the contiguous per-expert batches"
// of "Mixture of experts (MoE)" (tirogla.com), How it works step 4 and Implementation
// notes; the expert is the SwiGLU MLP of "DL S077 - Mixture of Experts (MoE) Intuition",
// section 1.1 (w1 = gate, w3 = up, w2 = down).
//
// Three epilogues share the main loop:
//   TC_SWIGLU : B tile = [W1 rows n0..n0+BN/2 ; W3 rows n0..n0+BN/2]; one MMA of width BN
//               gives gate and up side by side in TMEM; the epilogue writes
//               H = silu(gate) * up as bf16 (BN/2 output columns per tile).
//   TC_SCALE  : down projection; the epilogue writes g_r * acc as bf16, with the gate
//               g_r = topk_gate[perm[r]] of the row's assignment (1 for the shared expert).
//   TC_F32OUT : router logits (split-K planes); the epilogue writes acc as fp32.
//
// A CTA tile is MT x 128 rows by BN columns. With MT = 2 the B tile loaded for a k-block
// feeds two M=128 MMAs (rows r..r+127 and r+128..r+255), halving the weight bytes per FLOP
// that cross L2 and shared memory, so the 3-stage ring covers more latency than the
// 4-stage ring of MT = 1 (the kernel is bound by how many bytes it keeps in flight). The
// last row tile of a group may have only its first half valid: then the second half is
// neither loaded nor multiplied.
//
// Short row tiles (AR = 32, used when no group has more than 32 rows, e.g. a decode step):
// only 32 rows of A are loaded per k-block (4 KB instead of 16 KB), so more stages fit and
// more weight bytes stay in flight. The M=128 MMA still reads a 16 KB A window; its rows
// 32..127 are the bytes that follow inside the same stage (already landed), and the
// accumulator rows they produce are never stored.
//
// Roles (one CTA per SM, persistent over tiles):
//   warp 0 lane 0  TMA producer: A tiles 128 x 64 and a B tile BN x 64 (bf16, 128-byte
//                  swizzle) into a STAGES-deep shared-memory ring;
//   warp 1         allocates TMEM; lane 0 issues tcgen05.mma (M=128, N=BN, K=16). MT = 1
//                  keeps two accumulators so the epilogue of tile i overlaps the MMAs of
//                  i+1; MT = 2 uses all 512 columns for the two row halves;
//   warps 2..      epilogue, 4 warps per row half: tcgen05.ld (each warp reads its 32-lane
//                  quarter of TMEM), element-wise math, then a 16-bit output block of 32
//                  rows x CW columns is staged in shared memory (swizzled, two buffers per
//                  warp) and written by one TMA tensor store; a block that reaches past its
//                  group's end (A tiles may straddle two experts) is stored row by row with
//                  those rows masked;
//   (W8) 8 warps   converters: E4M3 weight tile in the TMA ring -> fp16 tile in a separate
//                  2-slot ring that the MMA reads, so the TMA ring holds only A and the
//                  8-bit staging and keeps more weight bytes in flight. The conversion is
//                  the 8-bit path's bottleneck, so it targets fp16 (one hardware
//                  conversion per weight pair, exact); bf16 operands would need a longer
//                  one. So the 8-bit path runs its MMAs on fp16 operands: the gather
//                  converts the activations to fp16 and the SwiGLU epilogue writes H as
//                  fp16.
// Every mbarrier wait is bounded (common.cuh): on a timeout the kernel records
// MOE_ERR_TIMEOUT in the workspace error word, drains its own copies and MMAs, frees TMEM
// and returns.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "launchers.h"
#include "tma_host.h"

namespace moe {

namespace {

constexpr int BM = 128;
constexpr int kMaxGroups = 1024;

__host__ __device__ constexpr uint32_t pow2_at_least(uint32_t v) {
  uint32_t p = 32;
  while (p < v) p <<= 1;
  return p;
}

// KB: K elements per pipeline stage -- 64 (128-byte rows, 128-byte swizzle) or 32 (64-byte
// rows, 64-byte swizzle: half the bytes per stage, twice the stages in flight).
// W8: the B operand arrives as E4M3 codes (one byte per element) in the TMA stage and
// CONV_WARPS converter warps expand it to fp16 in a slot of the conversion ring.
// AR: rows of A loaded per k-block, 128 or 32 (short row tiles, MT = 1 only).
template <int MODE, int BN, int MT, int KB, bool W8 = false, int AR = 128>
struct Cfg {
  static constexpr int BK = KB;
  static constexpr int SW = KB * 2;                     // swizzle span = bytes per row
  static constexpr int EPI_WARPS = 4 * MT;
  static constexpr int CONV_WARPS = W8 ? 8 : 0;
  static constexpr int THREADS = 64 + 32 * (EPI_WARPS + CONV_WARPS);
  static constexpr int TM = (AR < BM) ? AR : MT * BM;   // rows per CTA tile
  static constexpr int A_BYTES = AR * BK * 2;           // one A tile as loaded
  static constexpr int B_BYTES = BN * BK * 2;           // 16-bit B tile (the MMA operand)
  static constexpr int B8_BYTES = W8 ? BN * BK : 0;     // 8-bit B tile as loaded
  // TMA ring: A tile(s) then the B tile (bf16, or 8-bit for W8)
  static constexpr int STAGE_BYTES = MT * A_BYTES + (W8 ? B8_BYTES : B_BYTES);
  // conversion ring (W8): fp16 B tiles written by the converters, read by the MMA
  static constexpr int CSTAGES = W8 ? 2 : 0;
  static constexpr int CSTAGE_BYTES = W8 ? B_BYTES : 0;
  static constexpr int STAGES_RAW = (196 * 1024 - CSTAGES * CSTAGE_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 12 ? 12 : STAGES_RAW;
  static constexpr int BN_OUT = (MODE == TC_SWIGLU) ? BN / 2 : BN;
  static constexpr int NUM_ACC = (MT == 1) ? 2 : 1;    // accumulator sets (double buffering)
  static constexpr uint32_t TMEM_COLS = pow2_at_least(NUM_ACC * MT * BN);
  static constexpr uint32_t IDESC = W8 ? idesc_f16_f32(BM, BN) : idesc_bf16_f32(BM, BN);
  // epilogue chunk: output columns per TMEM read (SwiGLU: CW gate + CW up columns)
  static constexpr int CW = (MODE == TC_SWIGLU && BN_OUT % 32 != 0) ? 16 : 32;
  // 16-bit outputs leave through tensor stores: each epilogue warp stages 32 rows x CW
  // columns (CW * 2-byte rows, swizzled like the output map) in one of STG_BUFS buffers
  static constexpr int STG_ROW_BYTES = CW * 2;
  static constexpr int STG_BUF = 32 * STG_ROW_BYTES;
  static constexpr int STG_BUFS = 2;
  static constexpr int STG_BYTES = (MODE == TC_F32OUT) ? 0 : EPI_WARPS * STG_BUFS * STG_BUF;
  // shared memory layout (offsets from a 1024-byte aligned base)
  static constexpr int OFF_TILES = 0;
  static constexpr int OFF_CONV = STAGES * STAGE_BYTES;
  static constexpr int OFF_STG = OFF_CONV + CSTAGES * CSTAGE_BYTES;
  static constexpr int OFF_BARS = OFF_STG + STG_BYTES;
  // full, empty, tmem_full[2], tmem_empty[2], drain, converted[CSTAGES], conv_free[CSTAGES]
  static constexpr int NUM_BARS = 2 * STAGES + 5 + 2 * CSTAGES;
  static constexpr int OFF_MISC = OFF_BARS + NUM_BARS * 8;     // tmem slot, abort flag
  static constexpr int OFF_TABLE = OFF_MISC + 16;              // offsets[G+1], prefix[G+1]
  static constexpr int smem_bytes(int groups) {
    return 1024 + OFF_TABLE + 2 * (groups + 1) * 4;
  }
  static_assert(MT == 1 || MT == 2, "one or two 128-row tiles per CTA tile");
  static_assert(STAGES >= 2, "pipeline needs at least two stages");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "M=128 MMA needs N % 16 == 0, 16..256");
  static_assert(TMEM_COLS <= 512, "TMEM has 512 columns");
  static_assert((STAGE_BYTES % 1024) == 0, "stages must stay 1024-byte aligned");
  static_assert(KB == 64 || KB == 32, "64- or 32-element k-blocks");
  static_assert(!W8 || (MT == 1 && KB == 64), "8-bit weights use 128-row tiles, 64-wide k");
  static_assert(AR == BM || (MT == 1 && AR % 8 == 0 && AR >= 8), "short row tiles: MT = 1");
  static_assert(STAGE_BYTES >= BM * BK * 2, "the MMA's 128-row A window stays in its stage");
  static_assert((CSTAGE_BYTES % 1024) == 0, "conversion slots stay 1024-byte aligned");
  static_assert((STG_BUF % 1024) == 0, "staging buffers stay 1024-byte aligned (swizzle atoms)");
  static_assert(smem_bytes(1) <= kMaxDynSmem, "shared memory");
};

struct Tile {
  int shared;   // 1 = the shared-expert problem
  int group;    // expert (routed) or 0
  int n_blk;
  int row0;     // first row of A / output
  int rows;     // valid rows in this tile (<= MT * BM)
  int split;    // split-K index (router mode), else 0
  int kb0;      // first k-block (of BK) of this tile's K range
  int nk;       // k-blocks in the range
};

// Tile order inside a routed group: split fastest, then row tile, then column tile, so the
// CTAs that run at the same time share the group's weight tiles through L2.
template <int TM, int BK>
__device__ __forceinline__ Tile decode_tile(int tile, const int* s_off, const int* s_pre, int G,
                                            int nt_routed, int splits, const TcArgs& a) {
  Tile t;
  const int routed_total = s_pre[G];
  if (tile < routed_total) {
    int lo = 0, hi = G - 1;  // largest g with s_pre[g] <= tile
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_pre[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    const int g = lo;
    const int local = tile - s_pre[g];
    const int mt = (s_pre[g + 1] - s_pre[g]) / (nt_routed * splits);
    const int sp = local % splits;
    const int rest = local / splits;
    const int n = rest / mt, m = rest - n * mt;
    const int nk_all = (a.k_routed + BK - 1) / BK;
    t.shared = 0;
    t.group = g;
    t.n_blk = n;
    t.row0 = s_off[g] + m * TM;
    t.rows = min(TM, s_off[g + 1] - t.row0);
    t.split = sp;
    if (splits > 1) {
      t.kb0 = sp * a.kb_per_split;
      t.nk = min(nk_all - t.kb0, a.kb_per_split);
    } else {
      t.kb0 = 0;
      t.nk = nk_all;
    }
  } else {
    const int local = tile - routed_total;
    const int mt = (a.m_shared + TM - 1) / TM;
    const int n = local / mt, m = local - n * mt;
    t.shared = 1;
    t.group = 0;
    t.n_blk = n;
    t.row0 = m * TM;
    t.rows = min(TM, a.m_shared - t.row0);
    t.split = 0;
    t.kb0 = 0;
    t.nk = (a.k_shared + BK - 1) / BK;
  }
  return t;
}

template <int MODE, int BN, int MT, int KB, bool W8, int AR>
__global__ void __launch_bounds__(Cfg<MODE, BN, MT, KB, W8, AR>::THREADS, 1)
tc_grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB0,
                       const __grid_constant__ CUtensorMap tmB1,
                       const __grid_constant__ CUtensorMap tmAs,
                       const __grid_constant__ CUtensorMap tmB0s,
                       const __grid_constant__ CUtensorMap tmB1s,
                       const __grid_constant__ CUtensorMap tmO,
                       const __grid_constant__ CUtensorMap tmOs,
                       const __grid_constant__ CUtensorMap tmGU,
                       const __grid_constant__ CUtensorMap tmGUs, const TcArgs args) {
  using C = Cfg<MODE, BN, MT, KB, W8, AR>;
  constexpr int TM = C::TM;  // rows per CTA tile
  constexpr int BK = C::BK;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* tiles = smem + C::OFF_TILES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + C::STAGES;
  uint64_t* tfull_bar = bars + 2 * C::STAGES;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* drain_bar = tfull_bar + 4;
  uint64_t* conv_full = tfull_bar + 5;            // [CSTAGES], W8 only
  uint64_t* conv_empty = conv_full + C::CSTAGES;  // [CSTAGES], W8 only
  uint8_t* conv_tiles = smem + C::OFF_CONV;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  int* s_off = reinterpret_cast<int*>(smem + C::OFF_TABLE);
  const int G = args.groups;
  int* s_pre = s_off + (G + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  DeviceError* err = args.err;

  // ---- set-up: barriers (thread 0), TMEM (warp 1), group/tile tables (warp 2)
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], C::EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    for (int s = 0; s < C::CSTAGES; ++s) {
      mbar_init(&conv_full[s], C::CONV_WARPS);
      mbar_init(&conv_empty[s], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  // everything above touches only this CTA's own resources; from here on the kernel reads
  // what earlier kernels wrote (offsets, A)
  pdl_wait();
  pdl_launch_dependents();
  if (warp == 2) {
    // s_off[g] = first row of group g; s_pre[g] = first tile of group g (exclusive scan).
    const int nt = (args.n_routed + C::BN_OUT - 1) / C::BN_OUT * (MODE == TC_F32OUT ? args.splits : 1);
    int carry = 0;
    for (int base = 0; base < G; base += 32) {
      const int g = base + lane;
      int lo = 0, hi = 0;
      if (g < G) {
        if (args.offsets != nullptr) {
          lo = args.offsets[g];
          hi = args.offsets[g + 1];
        } else {
          lo = 0;
          hi = args.m_single;
        }
        s_off[g] = lo;
      }
      const int tiles_g = (g < G) ? ((hi - lo + TM - 1) / TM) * nt : 0;
      int incl = tiles_g;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (g < G) s_pre[g] = carry + incl - tiles_g;
      carry += __shfl_sync(0xffffffffu, incl, 31);
      if (g == G - 1) s_off[G] = hi;
    }
    if (lane == 0) s_pre[G] = carry;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int nt_routed = (args.n_routed + C::BN_OUT - 1) / C::BN_OUT;
  const int splits = (MODE == TC_F32OUT) ? args.splits : 1;
  const int nt_shared = args.has_shared ? (args.n_shared + C::BN_OUT - 1) / C::BN_OUT : 0;
  const int mt_shared = args.has_shared ? (args.m_shared + TM - 1) / TM : 0;
  const int total = s_pre[G] + mt_shared * nt_shared;

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB0);
      if (MODE == TC_SWIGLU) tma_prefetch_desc(&tmB1);
      if (args.has_shared) {
        tma_prefetch_desc(&tmAs);
        tma_prefetch_desc(&tmB0s);
        if (MODE == TC_SWIGLU) tma_prefetch_desc(&tmB1s);
      }
      uint32_t issued_mask = 0, parity_mask = 0;
      int stage = 0;
      uint32_t phase = 0;
      for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        const Tile t = decode_tile<TM, BK>(tile, s_off, s_pre, G, nt_routed, splits, args);
        const CUtensorMap* mA = t.shared ? &tmAs : &tmA;
        const CUtensorMap* mB0 = t.shared ? &tmB0s : &tmB0;
        const CUtensorMap* mB1 = t.shared ? &tmB1s : &tmB1;
        const bool two = (MT == 2) && (t.rows > BM);
        const uint32_t bytes = (W8 ? C::B8_BYTES : C::B_BYTES) + (two ? 2 : 1) * C::A_BYTES;
        bool ok = true;
        for (int kb = t.kb0; kb < t.kb0 + t.nk; ++kb) {
          if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1, abort_flag, err,
                                 SITE_GEMM_WAIT_EMPTY)) {
            ok = false;
            break;
          }
          uint8_t* sa = tiles + stage * C::STAGE_BYTES;
          uint8_t* sb = sa + MT * C::A_BYTES;
          mbar_arrive_expect_tx(&full_bar[stage], bytes);
          tma_load_2d(sa, mA, &full_bar[stage], kb * BK, t.row0);
          if (two) tma_load_2d(sa + C::A_BYTES, mA, &full_bar[stage], kb * BK, t.row0 + BM);
          if (MODE == TC_SWIGLU) {
            tma_load_3d(sb, mB0, &full_bar[stage], kb * BK, t.n_blk * (BN / 2), t.group);
            tma_load_3d(sb + (W8 ? C::B8_BYTES : C::B_BYTES) / 2, mB1, &full_bar[stage], kb * BK,
                        t.n_blk * (BN / 2), t.group);
          } else {
            tma_load_3d(sb, mB0, &full_bar[stage], kb * BK, t.n_blk * BN, t.group);
          }
          issued_mask |= 1u << stage;
          parity_mask = (parity_mask & ~(1u << stage)) | (phase << stage);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
      }
      // Drain: every copy this thread issued has landed before the CTA may exit.
      for (int s = 0; s < C::STAGES; ++s)
        if (issued_mask & (1u << s))
          mbar_wait_bounded(&full_bar[s], (parity_mask >> s) & 1u, nullptr, err,
                            SITE_GEMM_WAIT_DRAIN);
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      int stage = 0, cstage = 0;
      uint32_t phase = 0, cphase = 0;
      int it = 0;
      bool ok = true, issued_any = false;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
        const Tile t = decode_tile<TM, BK>(tile, s_off, s_pre, G, nt_routed, splits, args);
        const bool two = (MT == 2) && (t.rows > BM);
        const int acc = it % C::NUM_ACC;
        const uint32_t acc_phase = (it / C::NUM_ACC) & 1;
        if (!mbar_wait_bounded(&tempty_bar[acc], acc_phase ^ 1, abort_flag, err,
                               SITE_GEMM_WAIT_TMEM_EMPTY))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * MT * BN);
        for (int kb = 0; kb < t.nk; ++kb) {
          // W8: the converters waited for this stage's copies before filling the slot
          if (!mbar_wait_bounded(W8 ? &conv_full[cstage] : &full_bar[stage], W8 ? cphase : phase,
                                 abort_flag, err, SITE_GEMM_WAIT_FULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(tiles + stage * C::STAGE_BYTES);
          const uint32_t b_addr =
              W8 ? smem_u32(conv_tiles + cstage * C::CSTAGE_BYTES) : a_addr + MT * C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t bdesc = smem_desc_kmajor<C::SW>(b_addr + kk * 32);
            const uint32_t accumulate = (kb | kk) != 0 ? 1u : 0u;
            tc_mma_bf16(d_tmem, smem_desc_kmajor<C::SW>(a_addr + kk * 32), bdesc, C::IDESC,
                        accumulate);
            if (two)
              tc_mma_bf16(d_tmem + BN, smem_desc_kmajor<C::SW>(a_addr + C::A_BYTES + kk * 32),
                          bdesc, C::IDESC, accumulate);
          }
          issued_any = true;
          tc_commit(&empty_bar[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
          if (W8) {
            tc_commit(&conv_empty[cstage]);
            if (++cstage == C::CSTAGES) {
              cstage = 0;
              cphase ^= 1;
            }
          }
        }
        if (ok) tc_commit(&tfull_bar[acc]);
      }
      // Drain: all MMAs issued by this thread have completed before TMEM is freed.
      if (issued_any) {
        tc_commit(drain_bar);
        mbar_wait_bounded(drain_bar, 0, nullptr, err, SITE_GEMM_WAIT_DRAIN);
      }
    }
  } else if (W8 && warp >= 2 + C::EPI_WARPS) {
    // ================= converters (8-bit weights) =================
    // Expand the staged E4M3 B tile (row r at r*64 bytes) to fp16 in the 128-byte swizzled
    // layout the MMA reads (16-byte chunk j of row r at chunk j ^ (r % 8)).
    const int ct = threadIdx.x - (2 + C::EPI_WARPS) * 32;
    int stage = 0, cstage = 0;
    uint32_t phase = 0, cphase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const Tile t = decode_tile<TM, BK>(tile, s_off, s_pre, G, nt_routed, splits, args);
      bool ok = true;
      for (int kb = 0; kb < t.nk; ++kb) {
        if (!mbar_wait_bounded(&full_bar[stage], phase, abort_flag, err, SITE_GEMM_WAIT_FULL) ||
            !mbar_wait_bounded(&conv_empty[cstage], cphase ^ 1, abort_flag, err,
                               SITE_GEMM_WAIT_EMPTY)) {
          ok = false;
          break;
        }
        const uint8_t* s8 = tiles + stage * C::STAGE_BYTES + MT * C::A_BYTES;
        uint8_t* sb = conv_tiles + cstage * C::CSTAGE_BYTES;
        // 16-byte chunk q of the staged tile holds row q / 4, bytes 16 * (q % 4) ..; every
        // thread issues all its loads before converting, so several are in flight
        constexpr int CT = 32 * (C::CONV_WARPS > 0 ? C::CONV_WARPS : 1);
        constexpr int CHUNKS = BN * 4;
        constexpr int PER = (CHUNKS + CT - 1) / CT;
        uint4 v[PER];
#pragma unroll
        for (int j = 0; j < PER; ++j) {
          const int q = ct + j * CT;
          if (q < CHUNKS) v[j] = *reinterpret_cast<const uint4*>(s8 + q * 16);
        }
#pragma unroll
        for (int j = 0; j < PER; ++j) {
          const int q = ct + j * CT;
          if (q < CHUNKS) {
            const int r = q >> 2, c = 2 * (q & 3);
            const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
            uint32_t o[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              o[2 * i] = e4m3x2_to_f16x2<0>(w[i]);
              o[2 * i + 1] = e4m3x2_to_f16x2<1>(w[i]);
            }
            uint8_t* row = sb + r * 128;
            *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) << 4)) =
                make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(row + (((c + 1) ^ (r & 7)) << 4)) =
                make_uint4(o[4], o[5], o[6], o[7]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&conv_full[cstage]);
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1;
        }
        if (++cstage == C::CSTAGES) {
          cstage = 0;
          cphase ^= 1;
        }
      }
      if (!ok) break;
    }
  } else {
    // ================= epilogue (warps 2 .. 2 + 4*MT - 1) =================
    const int half = (warp - 2) >> 2;      // which 128-row half of the CTA tile
    const int quarter = warp & 3;          // TMEM lanes this warp may read: 32*quarter .. +31
    const int r_local = half * BM + quarter * 32 + lane;
    // this warp's two staging buffers and the count of tensor stores it has issued
    uint8_t* stg = smem + C::OFF_STG + (warp - 2) * C::STG_BUFS * C::STG_BUF;
    uint32_t n_stores = 0;
    // Rows leave through a tensor store when all 32 of the warp's rows belong to the tile:
    // the box is then inside the group (a tile's rows past its group's end are the next
    // expert's rows, so a partial block is stored row by row instead).
    auto store_rows16 = [&](const CUtensorMap* map, const uint32_t* packed, int col0,
                            long long row_first) {
      uint8_t* buf = stg + (n_stores % C::STG_BUFS) * C::STG_BUF;
      if (n_stores >= C::STG_BUFS) {
        // the store that last read `buf` is done
        if (lane == 0) {
          if (C::STG_BUFS == 2) bulk_wait_group_read1(); else bulk_wait_group_read0();
        }
        __syncwarp();
      }
      stage_row_swizzled<C::STG_ROW_BYTES>(buf, packed, lane);
      store_staged_2d(map, buf, col0, static_cast<int>(row_first), lane);
      ++n_stores;
    };
    int it = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      const int acc = it % C::NUM_ACC;
      const uint32_t acc_phase = (it / C::NUM_ACC) & 1;
      if (!mbar_wait_bounded(&tfull_bar[acc], acc_phase, abort_flag, err,
                             SITE_GEMM_WAIT_TMEM_FULL))
        break;
      tc_fence_after();
      const Tile t = decode_tile<TM, BK>(tile, s_off, s_pre, G, nt_routed, splits, args);
      // a half with no valid row was not multiplied this tile, and a warp whose 32 rows are
      // all past the tile's end has nothing to store: skip (warp-uniform)
      if (half * BM < t.rows && half * BM + quarter * 32 < t.rows) {
        const bool rvalid = r_local < t.rows;
        const long long row = static_cast<long long>(t.row0) + r_local;
        const int N = t.shared ? args.n_shared : args.n_routed;
        const long long ldo = t.shared ? args.ldo_shared : args.ldo_routed;
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                               static_cast<uint32_t>((acc * MT + half) * BN);
        const int col_base = t.n_blk * C::BN_OUT;

        const long long row_first = static_cast<long long>(t.row0) + half * BM + quarter * 32;
        const bool whole_block = half * BM + quarter * 32 + 32 <= t.rows;
        const bool tma_rows = whole_block && ((args.tma_out >> t.shared) & 1);
        const CUtensorMap* omap = t.shared ? &tmOs : &tmO;
        if (MODE == TC_SWIGLU) {
          __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(t.shared ? args.out_shared
                                                                          : args.out_routed);
          // chunks of CW columns of H: gate columns [c*CW, +CW) and up columns BN/2 later
          constexpr int CW = C::CW;
#pragma unroll 1
          for (int c = 0; c < C::BN_OUT / CW; ++c) {
            uint32_t g[CW], u[CW];
            if constexpr (CW == 32) {
              tmem_ld_32cols(tbase + c * CW, g);
              tmem_ld_32cols(tbase + BN / 2 + c * CW, u);
            } else {
              tmem_ld_16cols(tbase + c * CW, g);
              tmem_ld_16cols(tbase + BN / 2 + c * CW, u);
            }
            tmem_ld_wait();
            void* gu = t.shared ? args.gu_shared : args.gu_routed;
            if (gu != nullptr && !W8 && whole_block && ((args.tma_out >> (2 + t.shared)) & 1) &&
                col_base + c * CW + CW <= N) {
              // pre-activations for the backward pass, whole chunk of a whole block: G at
              // columns col0.., U at N + col0.. of the [rows, 2N] map, two tensor stores
              const int col0 = col_base + c * CW;
              uint32_t pg[CW / 2], pu[CW / 2];
#pragma unroll
              for (int i = 0; i < CW / 2; ++i) {
                pg[i] = pack_bf16x2(__uint_as_float(g[2 * i]), __uint_as_float(g[2 * i + 1]));
                pu[i] = pack_bf16x2(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1]));
              }
              const CUtensorMap* gmap = t.shared ? &tmGUs : &tmGU;
              store_rows16(gmap, pg, col0, row_first);
              store_rows16(gmap, pu, N + col0, row_first);
            } else if (rvalid && gu != nullptr && !W8) {
              // pre-activations for the backward pass: G | U as bf16 [rows, 2N]
              const int col0 = col_base + c * CW;
              __nv_bfloat16* gdst = static_cast<__nv_bfloat16*>(gu) + row * 2 * N + col0;
#pragma unroll
              for (int q = 0; q < CW / 8; ++q)
                if (col0 + q * 8 < N) {
                  uint32_t pg[4], pu[4];
#pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    pg[i] = pack_bf16x2(__uint_as_float(g[8 * q + 2 * i]),
                                        __uint_as_float(g[8 * q + 2 * i + 1]));
                    pu[i] = pack_bf16x2(__uint_as_float(u[8 * q + 2 * i]),
                                        __uint_as_float(u[8 * q + 2 * i + 1]));
                  }
                  *reinterpret_cast<uint4*>(gdst + q * 8) = make_uint4(pg[0], pg[1], pg[2], pg[3]);
                  *reinterpret_cast<uint4*>(gdst + N + q * 8) =
                      make_uint4(pu[0], pu[1], pu[2], pu[3]);
                }
            }
            if (rvalid && out != nullptr) {
              const int col0 = col_base + c * CW;
              if (W8) {
                // per-row weight scales of W1 and W3, applied before the SiLU
                const float* s1 = args.scale0 + static_cast<size_t>(t.group) * N + col0;
                const float* s3 = args.scale1 + static_cast<size_t>(t.group) * N + col0;
#pragma unroll
                for (int i = 0; i < CW; ++i) {
                  const bool in = col0 + i < N;
                  g[i] = __float_as_uint(__uint_as_float(g[i]) * (in ? __ldg(s1 + i) : 0.f));
                  u[i] = __float_as_uint(__uint_as_float(u[i]) * (in ? __ldg(s3 + i) : 0.f));
                }
              }
              uint32_t packed[CW / 2];
              bool out_of_range = false;
#pragma unroll
              for (int i = 0; i < CW / 2; ++i) {
                const float h0 = silu_fast(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
                const float h1 =
                    silu_fast(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
                if (W8) {
                  // H is the down projection's fp16 operand
                  out_of_range |= fabsf(h0) > kF16Max || fabsf(h1) > kF16Max;
                  packed[i] = pack_f16x2(h0, h1);
                } else {
                  packed[i] = pack_bf16x2(h0, h1);
                }
              }
              if (W8 && out_of_range)
                record_error(args.err, MOE_ERR_NONFINITE, SITE_F16_RANGE_H, static_cast<int>(row));
              if (tma_rows) {
                store_rows16(omap, packed, col0, row_first);
              } else {
                __nv_bfloat16* dst = out + row * ldo + col0;
#pragma unroll
                for (int q = 0; q < CW / 8; ++q)
                  if (col0 + q * 8 < N)
                    *reinterpret_cast<uint4*>(dst + q * 8) = make_uint4(
                        packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
              }
            }
          }
        } else if (MODE == TC_SCALE) {
          __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(t.shared ? args.out_shared
                                                                          : args.out_routed);
          float gscale = 1.0f;
          long long orow = row;   // output row: the tile row, or its token (scatter_rows)
          if (rvalid && !t.shared) {
            if (args.row_gate != nullptr) {
              gscale = args.row_gate[row];
            } else if (args.gate != nullptr || args.scatter_rows) {
              const int a = args.perm[row];
              if (args.gate != nullptr) gscale = args.gate[a];
              if (args.scatter_rows) orow = a;
            }
          }
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t v[32];
            tmem_ld_32cols(tbase + c * 32, v);
            tmem_ld_wait();
            if (rvalid) {
              const int col0 = col_base + c * 32;
              if (W8) {
                // per-row scale of W2 (one per output column of the down projection)
                const float* s2 = args.scale0 + static_cast<size_t>(t.group) * N + col0;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  v[i] = __float_as_uint(__uint_as_float(v[i]) *
                                         (col0 + i < N ? __ldg(s2 + i) : 0.f));
              }
              uint32_t packed[16];
#pragma unroll
              for (int i = 0; i < 16; ++i)
                packed[i] = pack_bf16x2(gscale * __uint_as_float(v[2 * i]),
                                        gscale * __uint_as_float(v[2 * i + 1]));
              if (tma_rows) {
                store_rows16(omap, packed, col0, row_first);
              } else {
                __nv_bfloat16* dst = out + orow * ldo + col0;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  if (col0 + q * 8 < N)
                    *reinterpret_cast<uint4*>(dst + q * 8) = make_uint4(
                        packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
              }
            }
          }
        } else {  // TC_F32OUT
          float* out = reinterpret_cast<float*>(args.out_routed) + t.split * args.split_stride;
#pragma unroll 1
          for (int c = 0; c < BN / 16; ++c) {
            uint32_t v[16];
            tmem_ld_16cols(tbase + c * 16, v);
            tmem_ld_wait();
            if (rvalid) {
              const int col0 = col_base + c * 16;
              float* dst = out + row * ldo + col0;
              if (args.bias == nullptr && col0 + 16 <= N && (ldo & 3) == 0) {
                // whole 16-column chunk inside the row: four 16-byte stores
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  *reinterpret_cast<uint4*>(dst + 4 * q) =
                      make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
              } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  const int col = col0 + i;
                  if (col < N) {
                    float val = __uint_as_float(v[i]);
                    if (args.bias != nullptr) val += args.bias[col];
                    dst[i] = val;
                  }
                }
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[acc]);
    }
    // this warp's tensor stores are complete before the CTA exits
    if (lane == 0 && n_stores > 0) bulk_wait_group0();
  }

  // ---- teardown: all roles are done with TMEM before it is freed
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------------------------
// Host side: tensor maps and launch
// ------------------------------------------------------------------------------------
template <int MODE, int BN, int MT, int KB, bool W8, int AR>
int launch_impl(const TcProblem& p, cudaStream_t stream) {
  using C = Cfg<MODE, BN, MT, KB, W8, AR>;
  if (!get_encoder()) return MOE_ERR_CUDA;
  const int groups = p.args.groups;
  if (groups < 1 || groups > kMaxGroups) return MOE_ERR_INVALID;
  const uint32_t brows = (MODE == TC_SWIGLU) ? BN / 2 : BN;

  CUtensorMap mA{}, mB0{}, mB1{}, mAs{}, mB0s{}, mB1s{};
  if (!encode_2d(&mA, p.a, p.args.k_routed, p.a_rows, AR, KB)) return MOE_ERR_CUDA;
  if (W8) {
    if (p.args.has_shared || p.args.scale0 == nullptr ||
        (MODE == TC_SWIGLU && p.args.scale1 == nullptr))
      return MOE_ERR_INVALID;
    if (!encode_3d_u8(&mB0, p.b0, p.args.k_routed, p.b_rows, p.b_groups, brows, KB))
      return MOE_ERR_CUDA;
    if (MODE == TC_SWIGLU &&
        !encode_3d_u8(&mB1, p.b1, p.args.k_routed, p.b_rows, p.b_groups, brows, KB))
      return MOE_ERR_CUDA;
  } else {
    if (!encode_3d(&mB0, p.b0, p.args.k_routed, p.b_rows, p.b_groups, brows, KB))
      return MOE_ERR_CUDA;
    if (MODE == TC_SWIGLU &&
        !encode_3d(&mB1, p.b1, p.args.k_routed, p.b_rows, p.b_groups, brows, KB))
      return MOE_ERR_CUDA;
  }
  if (p.args.has_shared) {
    if (!encode_2d(&mAs, p.a_s, p.args.k_shared, p.args.m_shared, AR, KB)) return MOE_ERR_CUDA;
    if (!encode_3d(&mB0s, p.b0_s, p.args.k_shared, p.b_rows_s, 1, brows, KB)) return MOE_ERR_CUDA;
    if (MODE == TC_SWIGLU && !encode_3d(&mB1s, p.b1_s, p.args.k_shared, p.b_rows_s, 1, brows, KB))
      return MOE_ERR_CUDA;
  }

  // 16-bit outputs through tensor stores where the buffers allow (16-byte aligned base and
  // row stride); otherwise the epilogue stores element-wise
  TcArgs args = p.args;
  args.tma_out = 0;
  CUtensorMap mO{}, mOs{};
  if (MODE == TC_SCALE && args.scatter_rows && (args.perm == nullptr || args.row_gate != nullptr))
    return MOE_ERR_INVALID;
  if (MODE != TC_F32OUT) {
    // routed rows scattered to their tokens are stored row by row
    if (!args.scatter_rows &&
        encode_2d_out16(&mO, args.out_routed, args.n_routed, p.a_rows, args.ldo_routed, C::CW))
      args.tma_out |= 1;
    if (args.has_shared &&
        encode_2d_out16(&mOs, args.out_shared, args.n_shared, args.m_shared, args.ldo_shared, C::CW))
      args.tma_out |= 2;
  }
  // the backward's pre-activations G | U [rows, 2N]: U starts at column N, so N % 8 == 0
  CUtensorMap mGU{}, mGUs{};
  if (MODE == TC_SWIGLU && !W8) {
    if (args.n_routed % 8 == 0 &&
        encode_2d_out16(&mGU, args.gu_routed, 2ull * args.n_routed, p.a_rows,
                        2ull * args.n_routed, C::CW))
      args.tma_out |= 4;
    if (args.has_shared && args.n_shared % 8 == 0 &&
        encode_2d_out16(&mGUs, args.gu_shared, 2ull * args.n_shared, args.m_shared,
                        2ull * args.n_shared, C::CW))
      args.tma_out |= 8;
  }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  const int smem = C::smem_bytes(groups);
  if (smem > kMaxDynSmem) return MOE_ERR_UNSUPPORTED;
  static std::once_flag attr_once[64];
  static bool attr_ok[64];
  if (dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::call_once(attr_once[dev], [&]() {
    attr_ok[dev] = cudaFuncSetAttribute(tc_grouped_gemm_kernel<MODE, BN, MT, KB, W8, AR>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        std::min(C::smem_bytes(kMaxGroups), kMaxDynSmem)) ==
                   cudaSuccess;
  });
  if (!attr_ok[dev]) return MOE_ERR_CUDA;

  long long grid = std::min<long long>(p.max_tiles, p.num_sms);
  if (grid < 1) return MOE_OK;
  if (launch_pdl(tc_grouped_gemm_kernel<MODE, BN, MT, KB, W8, AR>, dim3(static_cast<int>(grid)),
                 dim3(C::THREADS), smem, stream, mA, mB0, mB1, mAs, mB0s, mB1s, mO, mOs, mGU,
                 mGUs, args) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

static_assert(Cfg<TC_SWIGLU, 256, 2, 64>::smem_bytes(kTcMt2MaxGroups) <= kMaxDynSmem &&
                  Cfg<TC_SCALE, 256, 2, 64>::smem_bytes(kTcMt2MaxGroups) <= kMaxDynSmem,
              "256-row tiles fit up to kTcMt2MaxGroups groups");

}  // namespace

int launch_tc_gemm(int mode, int bn, int mt, int kb, bool w8, int ar, const TcProblem& p,
                   cudaStream_t stream) {
#define MOE_TC_CASE(M, N, T, K, W, R)                                             \
  if (mode == M && bn == N && mt == T && kb == K && w8 == (W != 0) && ar == R) \
    return launch_impl<M, N, T, K, W != 0, R>(p, stream);
  MOE_TC_CASE(TC_SWIGLU, 256, 1, 64, 0, 128)
  MOE_TC_CASE(TC_SWIGLU, 224, 1, 64, 0, 128)
  MOE_TC_CASE(TC_SWIGLU, 256, 2, 64, 0, 128)
  MOE_TC_CASE(TC_SWIGLU, 256, 1, 64, 0, 32)
  MOE_TC_CASE(TC_SWIGLU, 224, 1, 64, 0, 32)
  MOE_TC_CASE(TC_SCALE, 256, 1, 64, 0, 128)
  MOE_TC_CASE(TC_SCALE, 256, 2, 64, 0, 128)
  MOE_TC_CASE(TC_SCALE, 256, 1, 64, 0, 32)
  MOE_TC_CASE(TC_SWIGLU, 256, 1, 64, 1, 128)
  MOE_TC_CASE(TC_SWIGLU, 224, 1, 64, 1, 128)
  MOE_TC_CASE(TC_SWIGLU, 256, 1, 64, 1, 32)
  MOE_TC_CASE(TC_SWIGLU, 224, 1, 64, 1, 32)
  MOE_TC_CASE(TC_SCALE, 256, 1, 64, 1, 128)
  MOE_TC_CASE(TC_SCALE, 256, 1, 64, 1, 32)
  MOE_TC_CASE(TC_F32OUT, 16, 1, 64, 0, 128)
  MOE_TC_CASE(TC_F32OUT, 32, 1, 64, 0, 128)
  MOE_TC_CASE(TC_F32OUT, 64, 1, 64, 0, 128)
  MOE_TC_CASE(TC_F32OUT, 128, 1, 64, 0, 128)
  MOE_TC_CASE(TC_F32OUT, 256, 1, 64, 0, 128)
#undef MOE_TC_CASE
  return MOE_ERR_UNSUPPORTED;
}

}  // namespace moe
