// Backward-pass GEMMs of the MoE layer on the 5th-generation tensor cores (tcgen05 + TMEM +
// TMA), sm_103a.
//
// The forward expert is O = w2 (silu(w1 x) * w3 x) ("DL S077 - Mixture of Experts (MoE)
// Intuition", section 1.1), applied to each expert's contiguous batch of rows ("Mixture of
// experts (MoE)", tirogla.com, How it works, step 4) and weighted by the gate in the combine
// (step 5). With G = Xp W1^T, U = Xp W3^T, H = silu(G) U, the chain rule gives, per expert:
//
//   BW_DGRAD_H  dH_raw = dYp . W2            (dYp: the upstream gradient of the row's token)
//               dH = g dH_raw,  dG = dH U silu'(G),  dU = dH silu(G),  dg = sum_f dH_raw H
//               (one kernel: the MMA gives dH_raw, the epilogue does the rest and also
//               writes H for the weight gradient of w2)
//   BW_DGRAD_X  dXp = dG . W1 + dU . W3      (one K loop over [dG dU] and [W1; W3])
//   BW_WGRAD    dW1 = dG^T Xp, dW3 = dU^T Xp, dW2 = (g dYp)^T H, each summed over the rows
//               of one expert (K = that expert's row count, ragged)
//
// The same kernel computes the router's dx = dlogits . W_r (BW_DGRAD_X with one group) and
// dW_r = dlogits^T x (BW_WGRAD with one group), and the shared expert's gradients.
//
// Operands. Every product here reads at least one matrix along its contiguous dimension:
// W2 [d, F] as the B operand of dH_raw (N = F is contiguous), W1 / W3 [F, d] for dXp, and
// both operands of every weight gradient (the K dimension is the row index). Nothing is
// transposed in HBM: those tiles are loaded MN-major (TMA boxes of 64 contiguous elements x
// 64 K rows, 128-byte swizzle) and the MMA reads them with MN-major descriptors.
//
// Roles (one CTA per SM, persistent): warp 0 lane 0 issues TMA; warp 1 allocates TMEM and
// lane 0 issues tcgen05.mma (M = 128, N = BN, K = 16) into one of two accumulators; warps
// 2..9 are the epilogue, two per 32-lane quarter of TMEM (warp w reads lanes 32*(w % 4)..,
// one half of the columns). BW_WGRAD writes its fp32 tiles through shared memory with TMA
// tensor stores (a thread holds one output row, so direct stores would touch 32 rows per
// instruction), and adds warps 10..13:
// the last k-block of an expert may run past the expert's rows (into the next expert's rows
// or the rows past the end), so they zero those rows of both staged tiles before the MMA
// reads them. The MMA waits for them on such tail k-blocks only; they look at every k-block
// in order and the producer reuses a stage only after they have (so they never fall a ring
// cycle behind and never touch a stage that holds another k-block). Every mbarrier wait is bounded (common.cuh): on a timeout the kernel records
// MOE_ERR_TIMEOUT, drains its own copies and MMAs, frees TMEM and returns.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "launchers.h"
#include "tma_host.h"

namespace moe {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kMaxGroups = 1024;
constexpr int kChunk = 64 * 128;  // one MN-major TMA box: 64 K rows x 128 bytes
// BW_WGRAD tensor stores: blocks of 32 rows x kStgCols fp32 columns staged per epilogue warp
constexpr int kStgCols = 16;
constexpr int kStgBytes = 32 * kStgCols * 4;

// MT (BW_WGRAD only): 128-row output tiles per CTA tile, 1 or 2. With MT = 2 one B tile
// feeds two M = 128 MMAs (output rows m0.. and m0 + 128..), twice the MMA work per staged
// byte; the two accumulators fill TMEM, so the epilogue is not double-buffered.
template <int MODE, int BN, int MT = 1>
struct BCfg {
  static constexpr bool A_MN = (MODE == BW_WGRAD);
  static constexpr int EPI_WARPS = 8;    // two per TMEM lane quarter
  static constexpr int MASK_WARPS = (MODE == BW_WGRAD) ? 4 : 0;
  static constexpr int THREADS = 64 + 32 * (EPI_WARPS + MASK_WARPS);
  static constexpr int A_BYTES = MT * BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int NUM_ACC = (MT == 1) ? 2 : 1;   // accumulator sets (double buffering)
  // one staging block per epilogue warp for the tensor stores (BW_WGRAD: 32 x 16 fp32;
  // DGRAD: 32 x 32 bf16, the same 2 KB)
  static constexpr int STG_BYTES = EPI_WARPS * kStgBytes;
  static constexpr int STAGES_RAW = (212 * 1024 - STG_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  static constexpr int OFF_STG = STAGES * STAGE_BYTES;
  static constexpr uint32_t TMEM_COLS = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64
                                       : (2 * BN <= 128) ? 128 : (2 * BN <= 256) ? 256 : 512;
  static_assert(MT == 1 || (MT == 2 && MODE == BW_WGRAD && 2 * BN <= 512), "MT = 2: weight grads");
  static constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN) | idesc_major(A_MN, true);
  static constexpr int OFF_BARS = OFF_STG + STG_BYTES;
  // full, empty, ready (tail rows masked), seen (maskers done with the stage),
  // tmem_full[2], tmem_empty[2], drain
  static constexpr int NUM_BARS = 4 * STAGES + 5;
  static constexpr int OFF_MISC = OFF_BARS + NUM_BARS * 8;
  static constexpr int OFF_TABLE = OFF_MISC + 16;
  static constexpr int smem_bytes(int groups) { return 1024 + OFF_TABLE + 2 * (groups + 1) * 4; }
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "B tiles are whole 64-wide chunks");
  static_assert(STAGES >= 2, "pipeline needs at least two stages");
};

struct BTile {
  int group;
  int m_blk;    // DGRAD: row tile; WGRAD: output row tile (of M)
  int n_blk;
  int row0;     // DGRAD: first A row; WGRAD: first K row (the group's first row)
  int rows;     // DGRAD: valid rows of the tile; WGRAD: K rows of the group
  int nk;       // k-blocks
};

template <int MODE>
__device__ __forceinline__ BTile decode(int tile, const int* s_off, const int* s_pre, int G,
                                        int nt, int mt, const BwdArgs& a) {
  BTile t;
  if (MODE == BW_WGRAD) {
    const int per = mt * nt;
    t.group = tile / per;
    const int local = tile - t.group * per;
    t.m_blk = local / nt;
    t.n_blk = local - t.m_blk * nt;
    t.row0 = s_off[t.group];
    t.rows = s_off[t.group + 1] - t.row0;
    t.nk = (t.rows + BK - 1) / BK;
  } else {
    int lo = 0, hi = G - 1;  // largest g with s_pre[g] <= tile
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_pre[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    t.group = lo;
    const int local = tile - s_pre[lo];
    const int rt = (s_pre[lo + 1] - s_pre[lo]) / nt;  // row tiles of this group
    t.n_blk = local / rt;
    t.m_blk = local - t.n_blk * rt;
    t.row0 = s_off[lo] + t.m_blk * BM;
    t.rows = min(BM, s_off[lo + 1] - t.row0);
    t.nk = (a.K + BK - 1) / BK;
  }
  return t;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <int MODE, int BN, int MT>
__global__ void __launch_bounds__(BCfg<MODE, BN, MT>::THREADS, 1)
tc_bwd_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
              const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmO0,
              const __grid_constant__ CUtensorMap tmO1, const BwdArgs args) {
  using C = BCfg<MODE, BN, MT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + C::STAGES;
  uint64_t* ready_bar = bars + 2 * C::STAGES;
  uint64_t* seen_bar = bars + 3 * C::STAGES;
  uint64_t* tfull_bar = bars + 4 * C::STAGES;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* drain_bar = tfull_bar + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  int* s_off = reinterpret_cast<int*>(smem + C::OFF_TABLE);
  const int G = args.groups;
  int* s_pre = s_off + (G + 1);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  DeviceError* err = args.err;

  const int nt = (args.N + BN - 1) / BN;
  const int mt = (MODE == BW_WGRAD) ? (args.M + MT * BM - 1) / (MT * BM) : 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
      mbar_init(&ready_bar[s], C::MASK_WARPS > 0 ? C::MASK_WARPS : 1);
      mbar_init(&seen_bar[s], C::MASK_WARPS > 0 ? C::MASK_WARPS : 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], C::EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  if (warp == 2) {
    // s_off[g]: first row of group g; s_pre[g]: first tile of group g (DGRAD row tiling)
    int carry = 0;
    for (int base = 0; base < G; base += 32) {
      const int g = base + lane;
      int lo = 0, hi = 0;
      if (g < G) {
        lo = args.offsets ? args.offsets[g] : 0;
        hi = args.offsets ? args.offsets[g + 1] : args.m_single;
        s_off[g] = lo;
      }
      const int tiles_g = (g < G) ? ((hi - lo + BM - 1) / BM) * nt : 0;
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
  const int total = (MODE == BW_WGRAD) ? G * mt * nt : s_pre[G];

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB0);
      if (MODE == BW_DGRAD_X) tma_prefetch_desc(&tmB1);
      uint32_t issued_mask = 0, parity_mask = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const BTile t = decode<MODE>(tile, s_off, s_pre, G, nt, mt, args);
        for (int kb = 0; kb < t.nk; ++kb) {
          // BW_WGRAD: the maskers must have looked at the stage's previous contents too
          if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1, abort_flag, err,
                                 SITE_GEMM_WAIT_EMPTY) ||
              (MODE == BW_WGRAD && !mbar_wait_bounded(&seen_bar[stage], phase ^ 1, abort_flag,
                                                      err, SITE_GEMM_WAIT_EMPTY))) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * C::STAGE_BYTES;
          uint8_t* sb = sa + C::A_BYTES;
          mbar_arrive_expect_tx(&full_bar[stage], C::A_BYTES + C::B_BYTES);
          const int n0 = t.n_blk * BN;
          if (MODE == BW_WGRAD) {
            const int krow = t.row0 + kb * BK;
            const int m0 = t.m_blk * MT * BM;
#pragma unroll
            for (int c = 0; c < 2 * MT; ++c)
              tma_load_2d(sa + c * kChunk, &tmA, &full_bar[stage], m0 + 64 * c, krow);
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              tma_load_2d(sb + c * kChunk, &tmB0, &full_bar[stage], n0 + 64 * c, krow);
          } else {
            tma_load_2d(sa, &tmA, &full_bar[stage], kb * BK, t.row0);
            const int kg = kb * BK;
            const bool second = (MODE == BW_DGRAD_X) && kg >= args.k_split;
            const CUtensorMap* mb = second ? &tmB1 : &tmB0;
            const int kr = second ? kg - args.k_split : kg;
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              tma_load_3d(sb + c * kChunk, mb, &full_bar[stage], n0 + 64 * c, kr, t.group);
          }
          issued_mask |= 1u << stage;
          parity_mask = (parity_mask & ~(1u << stage)) | (phase << stage);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      for (int s = 0; s < C::STAGES; ++s)
        if (issued_mask & (1u << s))
          mbar_wait_bounded(&full_bar[s], (parity_mask >> s) & 1u, nullptr, err,
                            SITE_GEMM_WAIT_DRAIN);
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t ready_phase = 0;   // BW_WGRAD: phase bit per stage of ready_bar (tails only)
      int it = 0;
      bool ok = true, issued_any = false;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
        const BTile t = decode<MODE>(tile, s_off, s_pre, G, nt, mt, args);
        const int acc = it % C::NUM_ACC;
        const uint32_t acc_phase = (it / C::NUM_ACC) & 1;
        if (!mbar_wait_bounded(&tempty_bar[acc], acc_phase ^ 1, abort_flag, err,
                               SITE_GEMM_WAIT_TMEM_EMPTY))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * MT * BN);
        // MT = 2: the second 128 output rows exist only if they start below M
        const bool two = (MT == 2) && (t.m_blk * MT * BM + BM < args.M);
        for (int kb = 0; kb < t.nk; ++kb) {
          // a k-block with rows past the group's end waits for the maskers, the rest only
          // for the copies
          const bool tail = (MODE == BW_WGRAD) && (t.rows - kb * BK < BK);
          if (!mbar_wait_bounded(tail ? &ready_bar[stage] : &full_bar[stage],
                                 tail ? (ready_phase >> stage) & 1u : phase, abort_flag, err,
                                 SITE_GEMM_WAIT_FULL)) {
            ok = false;
            break;
          }
          if (tail) ready_phase ^= 1u << stage;
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t b_addr = a_addr + C::A_BYTES;
          // a ragged last k-block of a group: skip the 16-row slices wholly past its rows
          const int krows = (MODE == BW_WGRAD) ? min(BK, t.rows - kb * BK) : BK;
          const int slices = (krows + 15) / 16;
          for (int kk = 0; kk < slices; ++kk) {
            const uint64_t adesc = C::A_MN ? smem_desc_mn_sw128(a_addr + kk * 2048, kChunk)
                                           : smem_desc_kmajor<128>(a_addr + kk * 32);
            const uint64_t bdesc = smem_desc_mn_sw128(b_addr + kk * 2048, kChunk);
            tc_mma_bf16(d_tmem, adesc, bdesc, C::IDESC, (kb | kk) != 0 ? 1u : 0u);
            if (two)   // rows 128..255: A chunks 2 and 3, the same B tile
              tc_mma_bf16(d_tmem + BN, smem_desc_mn_sw128(a_addr + 2 * kChunk + kk * 2048, kChunk),
                          bdesc, C::IDESC, (kb | kk) != 0 ? 1u : 0u);
          }
          issued_any = true;
          tc_commit(&empty_bar[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (ok) tc_commit(&tfull_bar[acc]);  // also for nk == 0: arrives at once
      }
      if (issued_any) {
        tc_commit(drain_bar);
        mbar_wait_bounded(drain_bar, 0, nullptr, err, SITE_GEMM_WAIT_DRAIN);
      }
    }
  } else if (MODE == BW_WGRAD && warp >= 2 + C::EPI_WARPS) {
    // ================= row maskers (ragged K) =================
    // Zero K rows [krows, 16 * ceil(krows / 16)) of the A and B tiles of a group's last
    // k-block: the MMA reads them (whole 16-row slices) but they belong to another group or
    // lie past the matrix. A row is 128 contiguous bytes of its 64-wide chunk (the swizzle
    // only permutes 16-byte units inside the row).
    const int mt_id = threadIdx.x - (2 + C::EPI_WARPS) * 32;
    constexpr int NCHUNK = 2 * MT + BN / 64;
    int stage = 0;
    uint32_t phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const BTile t = decode<MODE>(tile, s_off, s_pre, G, nt, mt, args);
      bool ok = true;
      for (int kb = 0; kb < t.nk; ++kb) {
        if (!mbar_wait_bounded(&full_bar[stage], phase, abort_flag, err, SITE_GEMM_WAIT_FULL)) {
          ok = false;
          break;
        }
        const int krows = min(BK, t.rows - kb * BK);
        if (krows < BK) {
          const int kend = min(BK, (krows + 15) & ~15);
          uint8_t* st = smem + stage * C::STAGE_BYTES;  // A chunks then B chunks, contiguous
          const int per_row = 8;                         // 16-byte stores per row
          const int work = NCHUNK * (kend - krows) * per_row;
          for (int i = mt_id; i < work; i += 32 * C::MASK_WARPS) {
            const int q = i % per_row;
            const int rr = i / per_row;
            const int chunk = rr / (kend - krows);
            const int row = krows + rr % (kend - krows);
            *reinterpret_cast<uint4*>(st + chunk * kChunk + row * 128 + q * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ready_bar[stage]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&seen_bar[stage]);
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
    }
  } else {
    // ================= epilogue (warps 2..9) =================
    const int quarter = warp & 3;
    // MT = 1: the two warps of a quarter split the BN columns; MT = 2: they take the two
    // 128-row halves, all columns each
    const int chalf = (MT == 1) ? (warp - 2) >> 2 : 0;
    const int rhalf = (MT == 2) ? (warp - 2) >> 2 : 0;
    const int r_local = quarter * 32 + lane;
    constexpr int CPW = (MT == 1) ? BN / 64 : BN / 32;   // 32-column chunks per warp
    uint8_t* stg = smem + C::OFF_STG + (warp - 2) * kStgBytes;
    bool stg_busy = false;                     // a tensor store may still read `stg`
    // DGRAD: one 32-row x 32-column bf16 block staged in the output map's 64-byte swizzle
    // (16-byte unit q of row `lane` at q ^ (lane / 2 % 4)) and written by one tensor store
    auto stage_store = [&](const CUtensorMap* map, const uint32_t* packed, int col0,
                           long long row_first) {
      if (stg_busy) {
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
      }
      stage_row_swizzled<64>(stg, packed, lane);
      store_staged_2d(map, stg, col0, static_cast<int>(row_first), lane);
      stg_busy = true;
    };
    int it = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      const int acc = it % C::NUM_ACC;
      const uint32_t acc_phase = (it / C::NUM_ACC) & 1;
      if (!mbar_wait_bounded(&tfull_bar[acc], acc_phase, abort_flag, err,
                             SITE_GEMM_WAIT_TMEM_FULL))
        break;
      tc_fence_after();
      const BTile t = decode<MODE>(tile, s_off, s_pre, G, nt, mt, args);
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>((acc * MT + rhalf) * BN);
      const int n0 = t.n_blk * BN;
      const int N = args.N;
      if (MODE == BW_WGRAD) {
        const int m_blk0 = t.m_blk * MT * BM + rhalf * BM + quarter * 32;  // first output row
        if (m_blk0 < args.M) {
          const bool second = m_blk0 >= args.m_split;
          const int ym = second ? m_blk0 - args.m_split : m_blk0;
#pragma unroll 1
          for (int cc = 0; cc < CPW; ++cc) {
            const int c = chalf * CPW + cc;
            const int col0 = n0 + c * 32;
            if (col0 >= N) break;
            uint32_t v[32];
            if (t.nk > 0) {
              tmem_ld_32cols(tbase + c * 32, v);
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = 0u;   // a group with no rows: dW = 0
            }
#pragma unroll
            for (int part = 0; part < 32 / kStgCols; ++part) {
              if (col0 + part * kStgCols >= N) break;
              if (stg_busy) {
                if (lane == 0) bulk_wait_group_read0();
                __syncwarp();
              }
              // row `lane` of the 32-row block, kStgCols fp32 values from column part * kStgCols
              stage_row_swizzled<kStgCols * 4>(stg, v + part * kStgCols, lane);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_3d(second ? &tmO1 : &tmO0, stg, col0 + part * kStgCols, ym, t.group);
                bulk_commit_group();
              }
              stg_busy = true;
            }
          }
        }
      } else if (quarter * 32 < t.rows) {
        const bool rvalid = r_local < t.rows;
        const long long row = static_cast<long long>(t.row0) + r_local;
        // whole 32-row blocks of whole 32-column chunks leave through tensor stores
        const long long row_first = static_cast<long long>(t.row0) + quarter * 32;
        const bool tma_blk = args.tma_out && quarter * 32 + 32 <= t.rows;   // warp-uniform
        if (MODE == BW_DGRAD_X) {
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out);
#pragma unroll 1
          for (int cc = 0; cc < CPW; ++cc) {
            const int c = chalf * CPW + cc;
            uint32_t v[32];
            tmem_ld_32cols(tbase + c * 32, v);
            tmem_ld_wait();
            const int col0 = n0 + c * 32;
            if (rvalid && col0 < N) {
              uint32_t packed[16];
#pragma unroll
              for (int i = 0; i < 16; ++i)
                packed[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
              if (tma_blk && col0 + 32 <= N) {
                stage_store(&tmO0, packed, col0, row_first);
              } else {
                __nv_bfloat16* dst = out + row * args.ldo + col0;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  if (col0 + 8 * q < N)
                    *reinterpret_cast<uint4*>(dst + 8 * q) = make_uint4(
                        packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
              }
            }
          }
        } else {  // BW_DGRAD_H
          float g_r = 1.0f;
          if (rvalid && args.gate != nullptr)
            g_r = args.perm != nullptr ? args.gate[args.perm[row]] : args.gate[row];
          const __nv_bfloat16* gu = static_cast<const __nv_bfloat16*>(args.gu) + row * 2 * N;
          __nv_bfloat16* dgu = static_cast<__nv_bfloat16*>(args.dgu) + row * 2 * N;
          __nv_bfloat16* hrow = static_cast<__nv_bfloat16*>(args.h) + row * N;
          float dg = 0.0f;
#pragma unroll 1
          for (int cc = 0; cc < CPW; ++cc) {
            const int c = chalf * CPW + cc;
            uint32_t v[32];
            tmem_ld_32cols(tbase + c * 32, v);
            tmem_ld_wait();
            const int col0 = n0 + c * 32;
            if (rvalid && col0 < N) {
              const bool tma_chunk = tma_blk && col0 + 32 <= N;   // warp-uniform
              uint32_t dgp[16], dup[16], hp[16];                 // tma_chunk: the packed chunk
              // all of the chunk's G and U loads first (read-only), then the math and stores
              uint4 gqs[4], uqs[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                if (col0 + 8 * q < N) {
                  gqs[q] = __ldg(reinterpret_cast<const uint4*>(gu + col0 + 8 * q));
                  uqs[q] = __ldg(reinterpret_cast<const uint4*>(gu + N + col0 + 8 * q));
                }
              }
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                if (col0 + 8 * q >= N) continue;
                const uint4 gq = gqs[q];
                const uint4 uq = uqs[q];
                const uint32_t gw[4] = {gq.x, gq.y, gq.z, gq.w};
                const uint32_t uw[4] = {uq.x, uq.y, uq.z, uq.w};
                uint32_t dgw[4], duw[4], hw[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  float dgv[2], duv[2], hv[2];
#pragma unroll
                  for (int h = 0; h < 2; ++h) {
                    const float gz = h ? bf16_hi(gw[i]) : bf16_lo(gw[i]);
                    const float uz = h ? bf16_hi(uw[i]) : bf16_lo(uw[i]);
                    const float raw = __uint_as_float(v[8 * q + 2 * i + h]);
                    const float sg = __fdividef(1.0f, 1.0f + __expf(-gz));
                    const float si = gz * sg;                          // silu(G)
                    const float dsi = sg * (1.0f + gz * (1.0f - sg));  // silu'(G)
                    const float dh = g_r * raw;
                    hv[h] = si * uz;
                    dgv[h] = dh * uz * dsi;
                    duv[h] = dh * si;
                    dg = fmaf(raw, hv[h], dg);
                  }
                  dgw[i] = pack_bf16x2(dgv[0], dgv[1]);
                  duw[i] = pack_bf16x2(duv[0], duv[1]);
                  hw[i] = pack_bf16x2(hv[0], hv[1]);
                }
                if (tma_chunk) {
#pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    dgp[4 * q + i] = dgw[i];
                    dup[4 * q + i] = duw[i];
                    hp[4 * q + i] = hw[i];
                  }
                } else {
                  *reinterpret_cast<uint4*>(dgu + col0 + 8 * q) =
                      make_uint4(dgw[0], dgw[1], dgw[2], dgw[3]);
                  *reinterpret_cast<uint4*>(dgu + N + col0 + 8 * q) =
                      make_uint4(duw[0], duw[1], duw[2], duw[3]);
                  *reinterpret_cast<uint4*>(hrow + col0 + 8 * q) =
                      make_uint4(hw[0], hw[1], hw[2], hw[3]);
                }
              }
              if (tma_chunk) {
                // dG at column col0 and dU at N + col0 of dG | dU [rows, 2N], H at col0 of H
                stage_store(&tmO0, dgp, col0, row_first);
                stage_store(&tmO0, dup, N + col0, row_first);
                stage_store(&tmO1, hp, col0, row_first);
              }
            }
          }
          // one partial per row, column tile and column half: [rows][n_tiles][2]
          if (rvalid && args.dg_part != nullptr)
            args.dg_part[row * args.n_tiles + 2 * t.n_blk + chalf] = dg;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[acc]);
    }
    if (lane == 0 && stg_busy) bulk_wait_group0();   // tensor stores done before exit
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <int MODE, int BN, int MT>
int launch_impl(const BwdProblem& p, cudaStream_t stream) {
  using C = BCfg<MODE, BN, MT>;
  if (!get_encoder()) return MOE_ERR_CUDA;
  const int groups = p.args.groups;
  if (groups < 1 || groups > kMaxGroups) return MOE_ERR_INVALID;
  CUtensorMap mA{}, mB0{}, mB1{}, mO0{}, mO1{};
  if (MODE == BW_WGRAD) {
    if (!encode_2d_mn(&mA, p.a, p.a_inner, p.a_rows, p.a_inner)) return MOE_ERR_CUDA;
    if (!encode_2d_mn(&mB0, p.b0, p.b_inner, p.b_rows, p.b_inner)) return MOE_ERR_CUDA;
    mB1 = mB0;
    const int g = p.args.groups;
    if (p.args.m_split % 32 != 0 && p.args.m_split != p.args.M) return MOE_ERR_INVALID;
    if (!encode_3d_f32_store(&mO0, p.args.out, p.args.N, p.args.m_split, g, kStgCols))
      return MOE_ERR_CUDA;
    if (p.args.M > p.args.m_split) {
      if (!encode_3d_f32_store(&mO1, p.args.out1, p.args.N, p.args.M - p.args.m_split, g,
                               kStgCols))
        return MOE_ERR_CUDA;
    } else {
      mO1 = mO0;
    }
  } else {
    if (!encode_2d(&mA, p.a, p.args.K, p.a_rows, BM, BK)) return MOE_ERR_CUDA;
    if (!encode_3d_mn(&mB0, p.b0, p.b_inner, p.b_rows, p.b_groups)) return MOE_ERR_CUDA;
    if (MODE == BW_DGRAD_X && p.b1 != nullptr) {
      if (!encode_3d_mn(&mB1, p.b1, p.b_inner, p.b_rows, p.b_groups)) return MOE_ERR_CUDA;
    } else {
      mB1 = mB0;
    }
  }
  // DGRAD outputs through tensor stores where the buffers allow it (16-byte aligned bases and
  // row strides; dG | dU needs N % 8 == 0 for U's first column)
  BwdArgs args = p.args;
  args.tma_out = 0;
  const unsigned long long N = static_cast<unsigned long long>(p.args.N);
  if (MODE == BW_DGRAD_X && args.out != nullptr &&
      encode_2d_out16(&mO0, args.out, N, p.a_rows, args.ldo, 32))
    args.tma_out = 1;
  if (MODE == BW_DGRAD_H && N % 8 == 0 && args.dgu != nullptr && args.h != nullptr &&
      encode_2d_out16(&mO0, args.dgu, 2 * N, p.a_rows, 2 * N, 32) &&
      encode_2d_out16(&mO1, args.h, N, p.a_rows, N, 32))
    args.tma_out = 1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  static std::once_flag attr_once[64];
  static bool attr_ok[64];
  std::call_once(attr_once[dev], [&]() {
    attr_ok[dev] = cudaFuncSetAttribute(tc_bwd_kernel<MODE, BN, MT>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        C::smem_bytes(kMaxGroups)) == cudaSuccess;
  });
  if (!attr_ok[dev]) return MOE_ERR_CUDA;
  const long long grid = std::min<long long>(p.max_tiles, p.num_sms);
  if (grid < 1) return MOE_OK;
  tc_bwd_kernel<MODE, BN, MT><<<static_cast<int>(grid), C::THREADS, C::smem_bytes(groups), stream>>>(
      mA, mB0, mB1, mO0, mO1, MODE == BW_WGRAD ? p.args : args);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

int launch_bwd_gemm(int mode, int bn, int mt, const BwdProblem& p, cudaStream_t stream) {
#define MOE_BW_CASE(M, N, T) \
  if (mode == M && bn == N && mt == T) return launch_impl<M, N, T>(p, stream);
  MOE_BW_CASE(BW_DGRAD_H, 256, 1)
  MOE_BW_CASE(BW_DGRAD_X, 256, 1)
  MOE_BW_CASE(BW_WGRAD, 256, 1)
  MOE_BW_CASE(BW_WGRAD, 256, 2)
  MOE_BW_CASE(BW_DGRAD_H, 128, 1)
  MOE_BW_CASE(BW_DGRAD_X, 128, 1)
  MOE_BW_CASE(BW_WGRAD, 128, 1)
#undef MOE_BW_CASE
  return MOE_ERR_UNSUPPORTED;
}

}  // namespace moe
