// Grouped GEMM on CTA pairs (tcgen05 cta_group::2), sm_103a: the 256-row tiles of the
// expert GEMMs -- gate/up with the SwiGLU epilogue and the down projection with the gate
// scale ("Mixture of experts (MoE)", tirogla.com, How it works steps 4-5; the SwiGLU expert
// of "DL S077 - Mixture of Experts (MoE) Intuition", section 1.1) -- for layers whose experts
// average many rows (the Mixtral-shaped prefill layer).
//
// Why pairs. A 256 x 256 output tile per k-block needs 64 KB of operands (A 256 x 64, B
// 256 x 64); on one SM its fp32 accumulator fills all 512 TMEM columns, so the epilogue of a
// tile cannot overlap the MMAs of the next. A cluster of two CTAs on two SMs splits the
// tile: CTA r holds A rows 128r..128r+127 and B rows (N/2)r..(N/2)r+N/2-1 (32 KB per stage
// each, the same bytes per FLOP), one thread of CTA 0 issues M = 256 MMAs that read both
// CTAs' shared memory, and each CTA's TMEM receives its 128 rows of D -- 256 columns, so both
// CTAs keep two accumulators and the epilogue runs under the next tile's MMAs.
//
// Roles (per CTA, one CTA per SM, the pair persistent over pair tiles):
//   warp 0 lane 0   TMA producer: this CTA's A rows and B half into a 6-stage ring. Both
//                   CTAs' copies complete on CTA 0's full barrier of the stage, which
//                   expects the bytes of both;
//   warp 1          TMEM (512 columns in both CTAs, allocated by one warp in each); lane 0
//                   of CTA 0 issues the M = 256 MMAs and commits to the empty and
//                   accumulator-full barriers of both CTAs;
//   warps 2..9      epilogue, two warps per TMEM lane quarter splitting the columns; each CTA
//                   stores its 128 rows (32-row blocks staged in shared memory and written
//                   by TMA tensor stores, row by row where a block passes its group's end)
//                   and arrives on CTA 0's accumulator-empty barrier.
// Every mbarrier wait is bounded (2 s); the last step is a cluster barrier, so neither CTA
// leaves while the other may still touch its shared memory or TMEM.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "launchers.h"
#include "tma_host.h"

namespace moe {

namespace {

constexpr int PBM = 128;   // rows of the pair tile held by one CTA
constexpr int PBK = 64;    // K elements per stage (128-byte rows, 128-byte swizzle)
constexpr int kPairMaxGroups = 1024;

template <int MODE, int BN>
struct PCfg {
  static constexpr int EPI_WARPS = 8;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int TM = 2 * PBM;                    // rows per pair tile
  static constexpr int A_BYTES = PBM * PBK * 2;         // this CTA's rows of A
  static constexpr int B_BYTES = (BN / 2) * PBK * 2;    // this CTA's half of the B tile
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES_RAW = (196 * 1024) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 10 ? 10 : STAGES_RAW;
  static constexpr int BN_OUT = (MODE == TC_SWIGLU) ? BN / 2 : BN;
  static constexpr uint32_t TMEM_COLS = 2 * BN;        // two accumulators of BN columns
  static constexpr uint32_t IDESC = idesc_bf16_f32(2 * PBM, BN);
  // tensor-store staging: one buffer of 32 rows x 32 bf16 columns (64-byte rows, swizzled
  // like the output map) per epilogue warp
  static constexpr int STG_BUF = 32 * 64;
  static constexpr int OFF_STG = STAGES * STAGE_BYTES;
  static constexpr int OFF_BARS = OFF_STG + EPI_WARPS * STG_BUF;
  // full[STAGES], empty[STAGES], tmem_full[2], tmem_empty[2], drain
  static constexpr int NUM_BARS = 2 * STAGES + 5;
  static constexpr int OFF_MISC = OFF_BARS + NUM_BARS * 8;     // tmem slot, abort flag
  static constexpr int OFF_TABLE = OFF_MISC + 16;              // offsets[G+1], prefix[G+1]
  static constexpr int smem_bytes(int groups) { return 1024 + OFF_TABLE + 2 * (groups + 1) * 4; }
  static_assert(MODE == TC_SWIGLU || MODE == TC_SCALE, "pair tiles: gate/up or down");
  static_assert(BN == 256, "pair tiles are 256 x 256 (B split 128 + 128)");
  static_assert(TMEM_COLS <= 512, "TMEM has 512 columns");
  static_assert(STAGE_BYTES % 1024 == 0, "stages stay 1024-byte aligned");
  static_assert(STAGES >= 4, "pipeline depth");
  static_assert(smem_bytes(kPairMaxGroups) <= kMaxDynSmem, "shared memory");
};

struct PTile {
  int shared, group, n_blk, row0, rows, nk;
};

// Tile order inside a routed group: row tile fastest, then column tile (the pairs that run
// at the same time share the group's weight tiles through L2); the shared expert last.
__device__ __forceinline__ PTile pair_tile(int tile, const int* s_off, const int* s_pre, int G,
                                           int nt_routed, const TcArgs& a) {
  constexpr int TM = 2 * PBM;
  PTile t;
  const int routed_total = s_pre[G];
  if (tile < routed_total) {
    int lo = 0, hi = G - 1;  // largest g with s_pre[g] <= tile
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_pre[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    const int local = tile - s_pre[lo];
    const int mt = (s_pre[lo + 1] - s_pre[lo]) / nt_routed;
    const int n = local / mt, m = local - n * mt;
    t.shared = 0;
    t.group = lo;
    t.n_blk = n;
    t.row0 = s_off[lo] + m * TM;
    t.rows = min(TM, s_off[lo + 1] - t.row0);
    t.nk = (a.k_routed + PBK - 1) / PBK;
  } else {
    const int local = tile - routed_total;
    const int mt = (a.m_shared + TM - 1) / TM;
    const int n = local / mt, m = local - n * mt;
    t.shared = 1;
    t.group = 0;
    t.n_blk = n;
    t.row0 = m * TM;
    t.rows = min(TM, a.m_shared - t.row0);
    t.nk = (a.k_shared + PBK - 1) / PBK;
  }
  return t;
}

template <int MODE, int BN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PCfg<MODE, BN>::THREADS, 1)
tc_pair_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB0,
                    const __grid_constant__ CUtensorMap tmB1,
                    const __grid_constant__ CUtensorMap tmAs,
                    const __grid_constant__ CUtensorMap tmB0s,
                    const __grid_constant__ CUtensorMap tmB1s,
                    const __grid_constant__ CUtensorMap tmO,
                    const __grid_constant__ CUtensorMap tmOs, const TcArgs args) {
  using C = PCfg<MODE, BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + C::STAGES;
  uint64_t* tfull_bar = bars + 2 * C::STAGES;
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
  const uint32_t rank = cluster_ctarank();   // 0: issues the MMAs
  const int cl = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(cluster_count_x());

  // ---- set-up: barriers, TMEM (one warp in each CTA), then a cluster barrier so that no
  // CTA signals a barrier of its peer before the peer has initialised it
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full_bar[s], 1);    // CTA 0's: its producer's arrive + both CTAs' bytes
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], 2 * C::EPI_WARPS);  // both CTAs' epilogue warps (CTA 0's copy)
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
  cluster_sync_all();
  pdl_wait();
  pdl_launch_dependents();
  if (warp == 2) {
    const int nt = (args.n_routed + C::BN_OUT - 1) / C::BN_OUT;
    int carry = 0;
    for (int base = 0; base < G; base += 32) {
      const int g = base + lane;
      int lo = 0, hi = 0;
      if (g < G) {
        if (args.offsets != nullptr) {
          lo = args.offsets[g];
          hi = args.offsets[g + 1];
        } else {
          hi = args.m_single;
        }
        s_off[g] = lo;
      }
      const int tiles_g = (g < G) ? ((hi - lo + C::TM - 1) / C::TM) * nt : 0;
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
  const int nt_shared = args.has_shared ? (args.n_shared + C::BN_OUT - 1) / C::BN_OUT : 0;
  const int mt_shared = args.has_shared ? (args.m_shared + C::TM - 1) / C::TM : 0;
  const int total = s_pre[G] + mt_shared * nt_shared;

  if (warp == 0) {
    // ================= TMA producer (both CTAs) =================
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
      for (int tile = cl; tile < total; tile += ncl) {
        const PTile t = pair_tile(tile, s_off, s_pre, G, nt_routed, args);
        const CUtensorMap* mA = t.shared ? &tmAs : &tmA;
        // SwiGLU: CTA 0 holds the W1 rows of the tile (gate), CTA 1 the W3 rows (up);
        // down projection: each CTA holds half of the tile's W2 rows
        const CUtensorMap* mB = (MODE == TC_SWIGLU && rank == 1) ? (t.shared ? &tmB1s : &tmB1)
                                                                 : (t.shared ? &tmB0s : &tmB0);
        const int b_row = (MODE == TC_SWIGLU) ? t.n_blk * (BN / 2)
                                              : t.n_blk * BN + static_cast<int>(rank) * (BN / 2);
        bool ok = true;
        for (int kb = 0; kb < t.nk; ++kb) {
          if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1, abort_flag, err,
                                 SITE_GEMM_WAIT_EMPTY)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * C::STAGE_BYTES;
          uint8_t* sb = sa + C::A_BYTES;
          if (rank == 0) mbar_arrive_expect_tx(&full_bar[stage], 2 * C::STAGE_BYTES);
          const uint32_t fb = cluster_addr(&full_bar[stage], 0);
          // rows past the tile's end (or the tensor's) are loaded too (zero-filled past the
          // tensor): the M = 256 MMA reads both halves; their results are not stored
          tma_load_2d_pair(sa, mA, fb, kb * PBK, t.row0 + static_cast<int>(rank) * PBM);
          tma_load_3d_pair(sb, mB, fb, kb * PBK, b_row, t.group);
          issued_mask |= 1u << stage;
          parity_mask = (parity_mask & ~(1u << stage)) | (phase << stage);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
      }
      // Drain: every copy this thread issued has landed before the CTA may exit -- CTA 0
      // sees its full barriers complete; CTA 1's copies complete on CTA 0's barriers, so it
      // waits until the MMAs have consumed each stage it filled (its empty barriers).
      for (int s = 0; s < C::STAGES; ++s)
        if (issued_mask & (1u << s))
          mbar_wait_bounded(rank == 0 ? &full_bar[s] : &empty_bar[s], (parity_mask >> s) & 1u,
                            nullptr, err, SITE_GEMM_WAIT_DRAIN);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ================= MMA issuer (CTA 0) =================
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int tile = cl; tile < total && ok; tile += ncl, ++it) {
        const PTile t = pair_tile(tile, s_off, s_pre, G, nt_routed, args);
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!mbar_wait_bounded(&tempty_bar[acc], acc_phase ^ 1, abort_flag, err,
                               SITE_GEMM_WAIT_TMEM_EMPTY))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < t.nk; ++kb) {
          if (!mbar_wait_bounded(&full_bar[stage], phase, abort_flag, err, SITE_GEMM_WAIT_FULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t b_addr = a_addr + C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < PBK / 16; ++kk)
            tc_mma_bf16_pair(d_tmem, smem_desc_kmajor<128>(a_addr + kk * 32),
                             smem_desc_kmajor<128>(b_addr + kk * 32), C::IDESC,
                             (kb | kk) != 0 ? 1u : 0u);
          tc_commit_pair(&empty_bar[stage], 0x3);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (ok) tc_commit_pair(&tfull_bar[acc], 0x3);
      }
      // Drain: every MMA issued here (they write both CTAs' TMEM and read both CTAs' shared
      // memory) has completed before the final cluster barrier.
      tc_commit_pair(drain_bar, 0x1);
      mbar_wait_bounded(drain_bar, 0, nullptr, err, SITE_GEMM_WAIT_DRAIN);
    }
  } else {
    // ================= epilogue (warps 2..9 of both CTAs) =================
    const int quarter = warp & 3;           // TMEM lanes this warp may read: 32*quarter .. +31
    const int chalf = (warp - 2) >> 2;      // which half of the tile's columns
    const int r_local = static_cast<int>(rank) * PBM + quarter * 32 + lane;  // row in the tile
    // Full 32-row blocks leave through a tensor store from this warp's staging buffer (a
    // block reaching past its group's end -- the next expert's rows -- row by row instead).
    uint8_t* stg = smem + C::OFF_STG + (warp - 2) * C::STG_BUF;
    uint32_t n_stores = 0;
    auto store_rows16 = [&](const CUtensorMap* map, const uint32_t* packed, int col0,
                            long long row_first) {
      if (n_stores > 0) {
        if (lane == 0) bulk_wait_group_read0();   // the previous store has read the buffer
        __syncwarp();
      }
      stage_row_swizzled<64>(stg, packed, lane);
      store_staged_2d(map, stg, col0, static_cast<int>(row_first), lane);
      ++n_stores;
    };
    int it = 0;
    for (int tile = cl; tile < total; tile += ncl, ++it) {
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!mbar_wait_bounded(&tfull_bar[acc], acc_phase, abort_flag, err,
                             SITE_GEMM_WAIT_TMEM_FULL))
        break;
      tc_fence_after();
      const PTile t = pair_tile(tile, s_off, s_pre, G, nt_routed, args);
      if (static_cast<int>(rank) * PBM + quarter * 32 < t.rows) {   // warp-uniform
        const bool rvalid = r_local < t.rows;
        const long long row = static_cast<long long>(t.row0) + r_local;
        const int N = t.shared ? args.n_shared : args.n_routed;
        const long long ldo = t.shared ? args.ldo_shared : args.ldo_routed;
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                               static_cast<uint32_t>(acc * BN);
        const int col_base = t.n_blk * C::BN_OUT;
        constexpr int CPW = C::BN_OUT / 32 / 2;   // 32-column chunks per warp
        const long long row_first =
            static_cast<long long>(t.row0) + static_cast<int>(rank) * PBM + quarter * 32;
        const bool tma_rows = static_cast<int>(rank) * PBM + quarter * 32 + 32 <= t.rows &&
                              ((args.tma_out >> t.shared) & 1);
        const CUtensorMap* omap = t.shared ? &tmOs : &tmO;
        if (MODE == TC_SWIGLU) {
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(t.shared ? args.out_shared
                                                                    : args.out_routed);
          void* gu = t.shared ? args.gu_shared : args.gu_routed;
#pragma unroll 1
          for (int cc = 0; cc < CPW; ++cc) {
            const int c = chalf * CPW + cc;
            uint32_t g[32], u[32];
            tmem_ld_32cols(tbase + c * 32, g);              // gate: columns 0..BN/2-1
            tmem_ld_32cols(tbase + BN / 2 + c * 32, u);     // up: columns BN/2..BN-1
            tmem_ld_wait();
            const int col0 = col_base + c * 32;
            if (rvalid && gu != nullptr) {
              // pre-activations for the backward pass: G | U as bf16 [rows, 2N]
              __nv_bfloat16* gdst = static_cast<__nv_bfloat16*>(gu) + row * 2 * N + col0;
#pragma unroll
              for (int q = 0; q < 4; ++q)
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
              uint32_t packed[16];
#pragma unroll
              for (int i = 0; i < 16; ++i)
                packed[i] = pack_bf16x2(
                    silu_fast(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]),
                    silu_fast(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]));
              if (tma_rows) {
                store_rows16(omap, packed, col0, row_first);
              } else {
                __nv_bfloat16* dst = out + row * ldo + col0;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  if (col0 + q * 8 < N)
                    *reinterpret_cast<uint4*>(dst + q * 8) = make_uint4(
                        packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
              }
            }
          }
        } else {  // TC_SCALE
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(t.shared ? args.out_shared
                                                                    : args.out_routed);
          float gscale = 1.0f;
          if (rvalid && !t.shared) {
            if (args.row_gate != nullptr) gscale = args.row_gate[row];
            else if (args.gate != nullptr) gscale = args.gate[args.perm[row]];
          }
#pragma unroll 1
          for (int cc = 0; cc < CPW; ++cc) {
            const int c = chalf * CPW + cc;
            uint32_t v[32];
            tmem_ld_32cols(tbase + c * 32, v);
            tmem_ld_wait();
            const int col0 = col_base + c * 32;
            if (rvalid) {
              uint32_t packed[16];
#pragma unroll
              for (int i = 0; i < 16; ++i)
                packed[i] = pack_bf16x2(gscale * __uint_as_float(v[2 * i]),
                                        gscale * __uint_as_float(v[2 * i + 1]));
              if (tma_rows) {
                store_rows16(omap, packed, col0, row_first);
              } else {
                __nv_bfloat16* dst = out + row * ldo + col0;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  if (col0 + q * 8 < N)
                    *reinterpret_cast<uint4*>(dst + q * 8) = make_uint4(
                        packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(&tempty_bar[acc], 0);
    }
    if (lane == 0 && n_stores > 0) bulk_wait_group0();   // stores complete before exit
  }

  // ---- teardown: both CTAs are done with each other's shared memory and TMEM
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

template <int MODE, int BN>
int launch_pair_impl(const TcProblem& p, cudaStream_t stream) {
  using C = PCfg<MODE, BN>;
  if (!get_encoder()) return MOE_ERR_CUDA;
  const int groups = p.args.groups;
  if (groups < 1 || groups > kPairMaxGroups) return MOE_ERR_INVALID;
  const uint32_t brows = BN / 2;   // each CTA loads half of the tile's B rows

  CUtensorMap mA{}, mB0{}, mB1{}, mAs{}, mB0s{}, mB1s{};
  if (!encode_2d(&mA, p.a, p.args.k_routed, p.a_rows, PBM, PBK)) return MOE_ERR_CUDA;
  if (!encode_3d(&mB0, p.b0, p.args.k_routed, p.b_rows, p.b_groups, brows, PBK))
    return MOE_ERR_CUDA;
  if (MODE == TC_SWIGLU &&
      !encode_3d(&mB1, p.b1, p.args.k_routed, p.b_rows, p.b_groups, brows, PBK))
    return MOE_ERR_CUDA;
  if (p.args.has_shared) {
    if (!encode_2d(&mAs, p.a_s, p.args.k_shared, p.args.m_shared, PBM, PBK)) return MOE_ERR_CUDA;
    if (!encode_3d(&mB0s, p.b0_s, p.args.k_shared, p.b_rows_s, 1, brows, PBK)) return MOE_ERR_CUDA;
    if (MODE == TC_SWIGLU && !encode_3d(&mB1s, p.b1_s, p.args.k_shared, p.b_rows_s, 1, brows, PBK))
      return MOE_ERR_CUDA;
  }

  TcArgs args = p.args;
  if (args.scatter_rows) return MOE_ERR_UNSUPPORTED;   // rows stay in expert order here
  args.tma_out = 0;
  CUtensorMap mO{}, mOs{};
  if (encode_2d_out16(&mO, args.out_routed, args.n_routed, p.a_rows, args.ldo_routed, 32))
    args.tma_out |= 1;
  if (args.has_shared &&
      encode_2d_out16(&mOs, args.out_shared, args.n_shared, args.m_shared, args.ldo_shared, 32))
    args.tma_out |= 2;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  auto kernel = tc_pair_gemm_kernel<MODE, BN>;
  // per device: the shared-memory opt-in and how many pairs can be resident at once
  static std::once_flag once[64];
  static int max_pairs[64];
  std::call_once(once[dev], [&]() {
    max_pairs[dev] = 0;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::smem_bytes(kPairMaxGroups)) != cudaSuccess)
      return;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2 * static_cast<unsigned>(std::max(1, p.num_sms / 2)));
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::smem_bytes(kPairMaxGroups);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    max_pairs[dev] = n;
  });
  if (max_pairs[dev] < 1) return MOE_ERR_CUDA;

  const long long pairs = std::min<long long>(p.max_tiles, max_pairs[dev]);
  if (pairs < 1) return MOE_OK;
  const int smem = C::smem_bytes(groups);
  if (launch_pdl(kernel, dim3(static_cast<int>(2 * pairs)), dim3(C::THREADS), smem, stream, mA,
                 mB0, mB1, mAs, mB0s, mB1s, mO, mOs, args) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace

int launch_tc_pair_gemm(int mode, const TcProblem& p, cudaStream_t stream) {
  if (mode == TC_SWIGLU) return launch_pair_impl<TC_SWIGLU, 256>(p, stream);
  if (mode == TC_SCALE) return launch_pair_impl<TC_SCALE, 256>(p, stream);
  return MOE_ERR_UNSUPPORTED;
}

}  // namespace moe
