// Grouped expert GEMMs on block-scaled 8-bit / 4-bit operands (tcgen05.mma kind::mxf8f6f4).
//
// "Mixture of Experts (MoE)" (learn.starphix.com), Inference Optimization, Quantization:
// experts stored in 8 or 4 bits; "DL S077 - Mixture of Experts (MoE) Intuition", section
// 8.2: DeepSeek-V3 computes in FP8. "Mixture of experts (MoE)" (tirogla.com), How it works,
// step 4: one grouped GEMM over the contiguous per-expert batches.
//
// Operands: A = activation rows as E4M3 codes [rows, K] with one scale per 32 K values in
// tile atoms (mx_quant.cu); B = expert weights as E4M3 codes [E, N, K] or E2M1 codes packed
// two per byte [E, N, K / 2] (the even element in the low nibble), with scales in atoms
// [E][N / 128][K / 128][512] (byte (n % 32) * 16 + ((n % 128) / 32) * 4 + (k / 32) % 4 for
// weight row n and column k, holding s + 127 for the scale 2^s). The tensor cores apply the
// scales while multiplying; the accumulators are fp32 in tensor memory.
//   MX_SWIGLU: B tile = [W1 rows n..n+127 ; W3 rows n..n+127], N = 256: gate and up side by
//              side in TMEM; the epilogue computes H = silu(gate) * up per row and writes it
//              as the down projection's A operand: E4M3 codes [rows, d_ff] and tile atoms
//              of its block scales (the same row tiles).
//   MX_SCALE : B tile = W2 rows n..n+255; the epilogue writes g_r * acc as bf16 rows.
// A k-block is 128 K values: 128 bytes per row (4-bit weights are unpacked by TMA to one
// byte per value in shared memory, 16 values then 8 empty bytes), 128-byte swizzle, four
// MMAs of K = 32, each selecting its byte of the scale columns.
//
// Roles (one CTA per SM, persistent over tiles):
//   warp 0 lane 0  TMA producer: A tile (AR rows), B tile (256 rows), and the k-block's three
//                  512-byte scale atoms (bulk copies) into a ring of stages;
//   warp 1         allocates TMEM; lane 0 copies the stage's scale atoms into TMEM columns
//                  of their own per stage (tcgen05.cp, 32 lanes x 16 bytes replicated to the
//                  four lane quarters) and issues the four block-scaled MMAs. A stage's scale
//                  columns are rewritten only after its data was refilled, i.e. after the
//                  MMAs that read them completed;
//   warps 2..9     epilogue: two warps per 32-lane quarter of TMEM, each taking every other
//                  32-column chunk.
// One accumulator of 256 columns (the scale columns take the rest of TMEM), so a tile's
// epilogue does not overlap the next tile's MMAs. Every wait is bounded (common.cuh).
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "launchers.h"
#include "tma_host.h"

namespace moe {
namespace {

constexpr int MX_BM = 128;       // MMA M
constexpr int MX_BK = 128;       // K values per stage
constexpr int MX_BN = 256;       // MMA N
constexpr int MX_MAX_GROUPS = 1024;

template <int MODE, int AR>
struct MxCfg {
  static constexpr int A_BYTES = AR * MX_BK;
  static constexpr int B_BYTES = MX_BN * MX_BK;
  static constexpr int SF_BYTES = 3 * 512;
  static constexpr int STAGE_BYTES = (A_BYTES + B_BYTES + SF_BYTES + 1023) / 1024 * 1024;
  static constexpr int STAGES_RAW = (200 * 1024) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  static constexpr int EPI_WARPS = 8;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int TM = AR;                          // rows per tile
  static constexpr int BN_OUT = MODE == TC_SWIGLU ? 128 : 256;
  static constexpr int SF_COLS = 12;                     // per stage: A 4, B 8
  static constexpr int ACC_COLS = MX_BN;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int OFF_BARS = STAGES * STAGE_BYTES;
  // full, empty, tmem_full, tmem_empty, drain
  static constexpr int NUM_BARS = 2 * STAGES + 3;
  static constexpr int OFF_MISC = OFF_BARS + NUM_BARS * 8;
  static constexpr int OFF_TABLE = OFF_MISC + 16;        // offsets, tile prefix, row-tile prefix
  static constexpr int smem_bytes(int groups) { return 1024 + OFF_TABLE + 3 * (groups + 1) * 4; }
  // tensor-store staging after the table, where it fits: one buffer per epilogue warp of 32
  // rows x 32 outputs (H codes: 32-byte rows; bf16 rows: 64 bytes), swizzled like the map
  static constexpr int STG_ROW_BYTES = MODE == TC_SWIGLU ? 32 : 64;
  static constexpr int STG_BUF = 32 * STG_ROW_BYTES;
  static constexpr int stg_offset(int groups) {
    return (OFF_TABLE + 3 * (groups + 1) * 4 + 1023) / 1024 * 1024;
  }
  static constexpr int smem_bytes_stg(int groups) {
    return 1024 + stg_offset(groups) + EPI_WARPS * STG_BUF;
  }
  static_assert(AR == 128 || AR == 32, "128- or 32-row tiles");
  static_assert(STAGES >= 2, "at least two stages");
  static_assert(ACC_COLS + SF_COLS * STAGES <= 512, "TMEM holds the accumulator and the scales");
  static_assert(STAGE_BYTES >= MX_BM * MX_BK, "the MMA's 128-row A window stays in its stage");
};

struct MxTile {
  int group, m, n_blk, row0, rows;
};

template <int TM>
__device__ __forceinline__ MxTile mx_decode_tile(int tile, const int* s_off, const int* s_pre,
                                                 int G, int nt) {
  int lo = 0, hi = G - 1;  // largest g with s_pre[g] <= tile
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_pre[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  MxTile t;
  t.group = lo;
  const int local = tile - s_pre[lo];
  const int mt = (s_pre[lo + 1] - s_pre[lo]) / nt;
  t.n_blk = local / mt;
  t.m = local - t.n_blk * mt;
  t.row0 = s_off[lo] + t.m * TM;
  t.rows = min(TM, s_off[lo + 1] - t.row0);
  return t;
}

template <int MODE, int AR, int BFMT>
__global__ void __launch_bounds__(MxCfg<MODE, AR>::THREADS, 1)
tc_mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                  const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmO,
                  const MxArgs args) {
  using C = MxCfg<MODE, AR>;
  constexpr int TM = C::TM;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + C::STAGES;
  uint64_t* tfull_bar = bars + 2 * C::STAGES;
  uint64_t* tempty_bar = tfull_bar + 1;
  uint64_t* drain_bar = tfull_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const int G = args.groups;
  int* s_off = reinterpret_cast<int*>(smem + C::OFF_TABLE);  // [G + 1] row offsets
  int* s_pre = s_off + (G + 1);                               // [G + 1] first tile of group
  int* s_pt = s_pre + (G + 1);                                // [G + 1] first row tile of group

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  DeviceError* err = args.err;
  const int nt = args.n / C::BN_OUT;      // column tiles per group
  const int nkb = args.k / MX_BK;         // k-blocks
  const int ka = args.k / 128;            // scale atoms along K (= nkb)

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, C::EPI_WARPS);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  pdl_wait();
  pdl_launch_dependents();
  if (warp == 2) {
    int carry = 0, carry_pt = 0;
    for (int base = 0; base < G; base += 32) {
      const int g = base + lane;
      int lo = 0, hi = 0;
      if (g < G) {
        lo = args.offsets[g];
        hi = args.offsets[g + 1];
        s_off[g] = lo;
      }
      const int rt = (g < G) ? (hi - lo + TM - 1) / TM : 0;
      int incl = rt * nt, incl_pt = rt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        const int w = __shfl_up_sync(0xffffffffu, incl_pt, o);
        if (lane >= o) {
          incl += v;
          incl_pt += w;
        }
      }
      if (g < G) {
        s_pre[g] = carry + incl - rt * nt;
        s_pt[g] = carry_pt + incl_pt - rt;
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
      carry_pt += __shfl_sync(0xffffffffu, incl_pt, 31);
      if (g == G - 1) s_off[G] = hi;
    }
    if (lane == 0) {
      s_pre[G] = carry;
      s_pt[G] = carry_pt;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = s_pre[G];
  constexpr uint32_t SF_BASE = C::ACC_COLS;
  // Balanced persistent grid: the fewest CTAs that keep the largest per-CTA tile count (e.g.
  // 896 tiles on 148 SMs: 128 CTAs of 7 tiles, not 8 of 7 and 140 of 6 with a last round
  // that streams on 8 SMs); the rest stay idle. The weight-streaming tiles are bound by the
  // bytes each SM keeps in flight, so a full last round matters more than the idle SMs.
  const int per_cta = (total + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
  const int nctas = per_cta > 0 ? (total + per_cta - 1) / per_cta : 0;
  const int first_tile = static_cast<int>(blockIdx.x) < nctas ? static_cast<int>(blockIdx.x) : total;

  if (warp == 0) {
    // ================= producer =================
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB0);
      if (MODE == TC_SWIGLU) tma_prefetch_desc(&tmB1);
      uint32_t issued = 0, parity = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = first_tile; tile < total && ok; tile += nctas) {
        const MxTile t = mx_decode_tile<TM>(tile, s_off, s_pre, G, nt);
        const uint8_t* sfa = args.sfa + static_cast<size_t>(s_pt[t.group] + t.m) * ka * 512;
        const size_t nrow_atoms = static_cast<size_t>(args.n_rows / 128);   // weight atoms along N
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1, abort_flag, err,
                                 SITE_GEMM_WAIT_EMPTY)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * C::STAGE_BYTES;
          uint8_t* sb = sa + C::A_BYTES;
          uint8_t* ssf = sb + C::B_BYTES;
          uint64_t* fb = &full_bar[stage];
          // 4-bit weights count at their packed size (64 bytes per 128 values), although
          // they land unpacked (one byte per value) in shared memory
          mbar_arrive_expect_tx(fb, C::A_BYTES + (BFMT == 5 ? C::B_BYTES / 2 : C::B_BYTES) +
                                        C::SF_BYTES);
          tma_load_2d(sa, &tmA, fb, kb * MX_BK, t.row0);
          bulk_load(ssf, sfa + static_cast<size_t>(kb) * 512, 512, fb);
          if (MODE == TC_SWIGLU) {
            tma_load_3d(sb, &tmB0, fb, kb * MX_BK, t.n_blk * 128, t.group);
            tma_load_3d(sb + C::B_BYTES / 2, &tmB1, fb, kb * MX_BK, t.n_blk * 128, t.group);
            const size_t a0 = ((t.group * nrow_atoms + t.n_blk) * ka + kb) * 512;
            bulk_load(ssf + 512, args.sfb0 + a0, 512, fb);
            bulk_load(ssf + 1024, args.sfb1 + a0, 512, fb);
          } else {
            tma_load_3d(sb, &tmB0, fb, kb * MX_BK, t.n_blk * 256, t.group);
            const size_t a0 = ((t.group * nrow_atoms + 2 * t.n_blk) * ka + kb) * 512;
            bulk_load(ssf + 512, args.sfb0 + a0, 512, fb);
            bulk_load(ssf + 1024, args.sfb0 + a0 + static_cast<size_t>(ka) * 512, 512, fb);
          }
          issued |= 1u << stage;
          parity = (parity & ~(1u << stage)) | (phase << stage);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      for (int s = 0; s < C::STAGES; ++s)
        if (issued & (1u << s))
          mbar_wait_bounded(&full_bar[s], (parity >> s) & 1u, nullptr, err, SITE_GEMM_WAIT_DRAIN);
    }
  } else if (warp == 1) {
    // ================= scale copies + MMA issuer =================
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true, issued_any = false;
      for (int tile = first_tile; tile < total && ok; tile += nctas, ++it) {
        if (!mbar_wait_bounded(tempty_bar, (it & 1) ^ 1, abort_flag, err,
                               SITE_GEMM_WAIT_TMEM_EMPTY))
          break;
        tc_fence_after();
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(&full_bar[stage], phase, abort_flag, err, SITE_GEMM_WAIT_FULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t b_addr = a_addr + C::A_BYTES;
          const uint32_t sf_addr = b_addr + C::B_BYTES;
          const uint32_t sf_col = tmem_base + SF_BASE + stage * C::SF_COLS;
          tc_cp_scale_atom(sf_col, smem_desc_plain16(sf_addr));
          tc_cp_scale_atom(sf_col + 4, smem_desc_plain16(sf_addr + 512));
          tc_cp_scale_atom(sf_col + 8, smem_desc_plain16(sf_addr + 1024));
#pragma unroll
          for (int kk = 0; kk < MX_BK / 32; ++kk)
            tc_mma_mx(tmem_base, smem_desc_kmajor<128>(a_addr + kk * 32),
                      smem_desc_kmajor<128>(b_addr + kk * 32), idesc_mx(MX_BM, MX_BN, BFMT, kk),
                      sf_col, sf_col + 4, (kb | kk) != 0 ? 1u : 0u);
          issued_any = true;
          tc_commit(&empty_bar[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (ok) tc_commit(tfull_bar);
      }
      if (issued_any) {
        tc_commit(drain_bar);
        mbar_wait_bounded(drain_bar, 0, nullptr, err, SITE_GEMM_WAIT_DRAIN);
      }
    }
  } else {
    // ================= epilogue (warps 2..5) =================
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;        // which of the two warps of this lane quarter
    const int r_local = quarter * 32 + lane;
    // Full 32-row blocks leave through a tensor store from this warp's staging buffer (a
    // block reaching past its group's end -- the next expert's rows -- row by row instead).
    uint8_t* stg = smem + C::stg_offset(G) + (warp - 2) * C::STG_BUF;
    uint32_t n_stores = 0;
    auto store_block = [&](const uint32_t* words, int col0, long long row_first) {
      if (n_stores > 0) {
        if (lane == 0) bulk_wait_group_read0();   // the previous store has read the buffer
        __syncwarp();
      }
      stage_row_swizzled<C::STG_ROW_BYTES>(stg, words, lane);
      store_staged_2d(&tmO, stg, col0, static_cast<int>(row_first), lane);
      ++n_stores;
    };
    int it = 0;
    for (int tile = first_tile; tile < total; tile += nctas, ++it) {
      if (!mbar_wait_bounded(tfull_bar, it & 1, abort_flag, err, SITE_GEMM_WAIT_TMEM_FULL)) break;
      tc_fence_after();
      const MxTile t = mx_decode_tile<TM>(tile, s_off, s_pre, G, nt);
      const bool any = quarter * 32 < t.rows;   // warp-uniform
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
      constexpr int NCH = MODE == TC_SWIGLU ? 2 : 4;   // 32-column chunks: c = half + 2 j
      // EARLY: this warp's share of the accumulator -- 32 rows x 128 values -- goes to
      // registers first and the accumulator is released at once, so the next tile's MMAs run
      // under the element-wise math and the stores (measured faster for the SwiGLU epilogue
      // with 4-bit weights only; elsewhere the extra registers spill and it is slower).
      // Otherwise each chunk is read just before its math and the accumulator is released
      // after the last one.
      constexpr bool EARLY = MODE == TC_SWIGLU && BFMT == 5;
      constexpr int NLD = EARLY ? NCH : 1;             // chunks held in registers at once
      uint32_t v0[NLD][32], v1[MODE == TC_SWIGLU ? NLD : 1][32];
      auto load_chunk = [&](int c, uint32_t (&a)[32], uint32_t (&b)[32]) {
        tmem_ld_32cols(tbase + c * 32, a);                              // gate, or the output
        if (MODE == TC_SWIGLU) tmem_ld_32cols(tbase + 128 + c * 32, b); // up
      };
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar);
      };
      if (EARLY) {
        if (any) {
#pragma unroll
          for (int j = 0; j < NLD; ++j) load_chunk(half + 2 * j, v0[j], v1[MODE == TC_SWIGLU ? j : 0]);
          tmem_ld_wait();
        }
        release();
      }
      if (!any) {
        if (!EARLY) release();
        continue;
      }
      const bool rvalid = r_local < t.rows;
      const long long row = static_cast<long long>(t.row0) + r_local;
      const long long row_first = static_cast<long long>(t.row0) + quarter * 32;
      const bool tma_rows = args.tma_out && quarter * 32 + 32 <= t.rows;   // warp-uniform
      if (MODE == TC_SWIGLU) {
        // H = silu(gate) * up for 128 columns, quantized in blocks of 32 to E4M3
        uint8_t* hq = args.out_codes + row * args.n + t.n_blk * 128;
        uint8_t* atom = args.out_atoms +
                        (static_cast<size_t>(s_pt[t.group] + t.m) * (args.n / 128) + t.n_blk) * 512 +
                        (r_local & 31) * 16 + (r_local >> 5) * 4;
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          const int c = half + 2 * j;
          const int jl = EARLY ? j : 0;
          if (!EARLY) {
            load_chunk(c, v0[0], v1[0]);
            tmem_ld_wait();
          }
          uint32_t w[8];
          int s = -127;
          if (rvalid) {
            float h[32];
#pragma unroll
            for (int i = 0; i < 32; ++i)
              h[i] = silu_fast(__uint_as_float(v0[jl][i])) * __uint_as_float(v1[jl][i]);
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(h[i]));
            if (!isfinite(amax)) {
              record_error(err, MOE_ERR_NONFINITE, SITE_MX_NONFINITE_H, static_cast<int>(row));
              amax = 0.f;
            }
            if (amax > 0.f) {
              int e;
              const float f = frexpf(amax, &e);
              s = max(-127, min(127, e - 9 + (f > 0.875f ? 1 : 0)));
            }
            const float mul = __int_as_float((127 - s) << 23);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              uint16_t a2, b2;
              asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
                  : "=h"(a2) : "f"(h[4 * i + 1] * mul), "f"(h[4 * i] * mul));
              asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
                  : "=h"(b2) : "f"(h[4 * i + 3] * mul), "f"(h[4 * i + 2] * mul));
              w[i] = static_cast<uint32_t>(a2) | (static_cast<uint32_t>(b2) << 16);
            }
          }
          if (tma_rows) {
            store_block(w, t.n_blk * 128 + c * 32, row_first);
          } else if (rvalid) {
            *reinterpret_cast<uint4*>(hq + c * 32) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(hq + c * 32 + 16) = make_uint4(w[4], w[5], w[6], w[7]);
          }
          if (rvalid) atom[c] = static_cast<uint8_t>(s + 127);
        }
      } else {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(args.out_rows);
        float gscale = 1.0f;
        if (rvalid) {
          if (args.row_gate != nullptr) gscale = args.row_gate[row];
          else if (args.gate != nullptr) gscale = args.gate[args.perm[row]];
        }
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          const int c = half + 2 * j;
          const int jl = EARLY ? j : 0;
          if (!EARLY) {
            load_chunk(c, v0[0], v1[0]);
            tmem_ld_wait();
          }
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            packed[i] = pack_bf16x2(gscale * __uint_as_float(v0[jl][2 * i]),
                                    gscale * __uint_as_float(v0[jl][2 * i + 1]));
          if (tma_rows) {
            store_block(packed, t.n_blk * 256 + c * 32, row_first);
          } else if (rvalid) {
            __nv_bfloat16* dst = out + row * args.ldo + t.n_blk * 256 + c * 32;
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<uint4*>(dst + q * 8) = make_uint4(
                  packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
          }
        }
      }
      if (!EARLY) release();
    }
    if (lane == 0 && n_stores > 0) bulk_wait_group0();   // stores complete before exit
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <int MODE, int AR, int BFMT>
int launch_mx_impl(const MxProblem& p, cudaStream_t stream) {
  using C = MxCfg<MODE, AR>;
  if (!get_encoder()) return MOE_ERR_CUDA;
  const int G = p.args.groups;
  if (G < 1 || G > MX_MAX_GROUPS) return MOE_ERR_INVALID;
  const int brows = MODE == TC_SWIGLU ? 128 : 256;
  CUtensorMap mA{}, mB0{}, mB1{};
  if (!encode_2d_u8_sw128(&mA, p.a, p.args.k, p.a_rows, AR)) return MOE_ERR_CUDA;
  if (BFMT == 5) {
    if (!encode_3d_e2m1_sw128(&mB0, p.b0, p.args.k, p.args.n_rows, G, brows)) return MOE_ERR_CUDA;
    if (MODE == TC_SWIGLU &&
        !encode_3d_e2m1_sw128(&mB1, p.b1, p.args.k, p.args.n_rows, G, brows))
      return MOE_ERR_CUDA;
  } else {
    if (!encode_3d_u8_sw128(&mB0, p.b0, p.args.k, p.args.n_rows, G, brows)) return MOE_ERR_CUDA;
    if (MODE == TC_SWIGLU && !encode_3d_u8_sw128(&mB1, p.b1, p.args.k, p.args.n_rows, G, brows))
      return MOE_ERR_CUDA;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  auto kernel = tc_mx_gemm_kernel<MODE, AR, BFMT>;
  static std::once_flag once[64];
  static bool attr_ok[64];
  // the outputs through tensor stores when the staging fits beside this layer's tile table
  MxArgs args = p.args;
  CUtensorMap mO{};
  args.tma_out = 0;
  int smem = C::smem_bytes(G);
  if (C::smem_bytes_stg(G) <= kMaxDynSmem) {
    const bool enc = MODE == TC_SWIGLU
                         ? encode_2d_out8(&mO, args.out_codes, args.n, p.a_rows, args.n)
                         : encode_2d_out16(&mO, args.out_rows, args.n, p.a_rows, args.ldo, 32);
    if (enc) {
      args.tma_out = 1;
      smem = C::smem_bytes_stg(G);
    }
  }
  std::call_once(once[dev], [&]() {
    attr_ok[dev] = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kMaxDynSmem) == cudaSuccess;
  });
  if (!attr_ok[dev]) return MOE_ERR_CUDA;
  const long long grid = std::min<long long>(p.max_tiles, p.num_sms);
  if (grid < 1) return MOE_OK;
  if (launch_pdl(kernel, dim3(static_cast<unsigned>(grid)), dim3(C::THREADS), smem, stream, mA,
                 mB0, mB1, mO, args) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace

int launch_mx_gemm(int mode, int ar, int bfmt, const MxProblem& p, cudaStream_t stream) {
#define MOE_MX_CASE(M, R, F) \
  if (mode == M && ar == R && bfmt == F) return launch_mx_impl<M, R, F>(p, stream);
  MOE_MX_CASE(TC_SWIGLU, 128, 0)
  MOE_MX_CASE(TC_SWIGLU, 32, 0)
  MOE_MX_CASE(TC_SWIGLU, 128, 5)
  MOE_MX_CASE(TC_SWIGLU, 32, 5)
  MOE_MX_CASE(TC_SCALE, 128, 0)
  MOE_MX_CASE(TC_SCALE, 32, 0)
  MOE_MX_CASE(TC_SCALE, 128, 5)
  MOE_MX_CASE(TC_SCALE, 32, 5)
#undef MOE_MX_CASE
  return MOE_ERR_UNSUPPORTED;
}

}  // namespace moe
