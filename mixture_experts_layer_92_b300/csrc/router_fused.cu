// The fused router: score and select in one kernel, the logits never leaving the chip.
//
// "Mixture of experts (MoE)" (tirogla.com), How it works, steps 1-2: the router computes
// l_t = x_t . W_r^T and each token keeps the top-k experts under the layer's gate
// convention; Implementation notes: the router's arithmetic is kept in fp32 (here: bf16
// operands, fp32 accumulation in tensor memory, fp32 logits); Complexity and constants: the
// router costs 2*T*d*E FLOPs, so it is bound by reading x, not by the tensor cores.
//
// One thread-block cluster of CS CTAs owns a tile of 128 tokens. CTA r of the cluster
// multiplies the tile's x rows by W_r over its own slice of the model width d (split K), so
// CS CTAs stream the tile's x at once and T/128 tiles fill the chip (one CTA per SM):
//   warp 0   TMA producer: x tile [128 x 64] and W_r tile [BN x 64] (bf16, 128-byte swizzle)
//            into a ring of stages;
//   warp 1   allocates TMEM; one thread issues tcgen05.mma (M = 128, N = BN >= E, K = 16)
//            accumulating the tile's partial logits in TMEM;
//   then all 16 warps drain TMEM (tcgen05.ld; warp w reads lane quarter w % 4) into a
//   [128 x E] fp32 block of shared memory (the ring's space, free once the MMAs are done).
// After a cluster barrier, CTA r finishes the logits of rows [r*128/CS, (r+1)*128/CS): its
// warps add, per token, the CS partial rows read from the cluster's shared memory
// (distributed shared memory) in rank order -- a fixed order, so the logits are
// bit-reproducible -- add the router bias, and run the routing step (route_token.cuh:
// softmax over all E, lse, top-k with ties to the lower index, gates) on several tokens per
// warp at once. Per-CTA sums of the probabilities and of lse^2 go to `partials` for the
// balance losses. A second cluster barrier keeps every CTA's shared memory alive until its
// peers have read it. Every mbarrier wait is bounded; on a timeout the kernel records
// MOE_ERR_TIMEOUT, still reaches both cluster barriers (its peers wait there) and frees its
// TMEM.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "launchers.h"
#include "route_token.cuh"
#include "tma_host.h"

namespace moe {
namespace {

constexpr int RF_BM = 128;        // tokens per cluster tile (the MMA's M)
constexpr int RF_BK = 64;         // K elements per stage: 128-byte rows, 128-byte swizzle
constexpr int RF_WARPS = 16;
constexpr int RF_THREADS = RF_WARPS * 32;
constexpr int RF_MAX_STAGES = 8;

struct RfArgs {
  int T, E, d;
  int kb_per;               // k-blocks (of 64) per CTA of a cluster
  int stages;               // ring depth
  int cs;                   // CTAs per cluster
  const float* bias;        // [E] or nullptr
  const float* select_bias; // [E] or nullptr (selection only)
  float* logits_out;        // [T][E] or nullptr
  float* probs_t;           // [E][T] or nullptr
  int k, gate_mode;
  int32_t* topk_idx;
  float* topk_gate;
  float* partials;          // [E + 1][gridDim.x]
  DeviceError* err;
};

template <int BN>
struct RfCfg {
  static constexpr int A_BYTES = RF_BM * RF_BK * 2;
  static constexpr int B_BYTES = BN * RF_BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t TMEM_COLS = BN < 32 ? 32 : BN;
  // partial logits in shared memory: row stride BN + 8 floats puts the rows that the lane
  // groups of a warp read at once (8 lanes x 4 rows) on distinct banks
  static constexpr int PSTRIDE = BN + 8;
  static constexpr int PART_BYTES = RF_BM * PSTRIDE * 4;
  static constexpr uint32_t IDESC = idesc_bf16_f32(RF_BM, BN);
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "M=128 MMA needs N % 16 == 0, 16..256");
  static_assert(STAGE_BYTES % 1024 == 0, "stages stay 1024-byte aligned");
  // bytes after the tile region (ring, later partial logits): per-warp statistics, then the
  // barriers and the TMEM slot
  __host__ __device__ static int stat_bytes(int E) { return RF_WARPS * (E + 1) * 4; }
  __host__ __device__ static int tile_bytes(int stages) {
    return stages * STAGE_BYTES > PART_BYTES ? stages * STAGE_BYTES : PART_BYTES;
  }
  // the deepest ring the shared memory holds (192 KB of stages)
  __host__ __device__ static constexpr int max_stages() {
    return (192 * 1024 / STAGE_BYTES) < RF_MAX_STAGES ? 192 * 1024 / STAGE_BYTES : RF_MAX_STAGES;
  }
  __host__ __device__ static int smem_bytes(int stages, int E) {
    return 1024 + tile_bytes(stages) + stat_bytes(E) + (2 * RF_MAX_STAGES + 2) * 8 + 16;
  }
};

// Loads a 32-bit word of CTA `rank`'s shared memory at this CTA's offset `p`.
__device__ __forceinline__ float ld_cluster_f32(const float* p, uint32_t rank) {
  float v;
  asm volatile(
      "{\n\t.reg .b32 ra;\n\t"
      "mapa.shared::cluster.u32 ra, %1, %2;\n\t"
      "ld.shared::cluster.f32 %0, [ra];\n\t}"
      : "=f"(v)
      : "r"(smem_u32(p)), "r"(rank)
      : "memory");
  return v;
}

template <int BN, int G, int J, int NT, bool FULL>
__global__ void __launch_bounds__(RF_THREADS, 1)
router_fused_kernel(const __grid_constant__ CUtensorMap tmX,
                    const __grid_constant__ CUtensorMap tmW, const RfArgs a) {
  using C = RfCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tile_bytes = C::tile_bytes(a.stages);
  uint8_t* ring = smem;
  float* part = reinterpret_cast<float*>(smem);  // after the MMAs: [128][PSTRIDE]
  float* s_stat = reinterpret_cast<float*>(smem + tile_bytes);  // [RF_WARPS][E + 1]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + tile_bytes + C::stat_bytes(a.E));
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + RF_MAX_STAGES;
  uint64_t* tfull_bar = bars + 2 * RF_MAX_STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * RF_MAX_STAGES + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int row0 = static_cast<int>(blockIdx.x / a.cs) * RF_BM;
  const int nk_all = (a.d + RF_BK - 1) / RF_BK;
  const int kb0 = static_cast<int>(rank) * a.kb_per;
  const int nk = max(0, min(a.kb_per, nk_all - kb0));
  DeviceError* err = a.err;

  // Set-up. Thread 0 (the TMA producer) initialises the barriers and issues the first ring's
  // worth of loads at once (every stage starts free), so the first bytes of x are on their
  // way while warp 1 allocates TMEM.
  int stage = 0;
  uint32_t phase = 0, issued = 0, parity = 0;
  int kb_issued = 0;
  auto issue = [&](int kb) {
    uint8_t* sa = ring + stage * C::STAGE_BYTES;
    mbar_arrive_expect_tx(&full_bar[stage], C::STAGE_BYTES);
    tma_load_2d(sa, &tmX, &full_bar[stage], (kb0 + kb) * RF_BK, row0);
    tma_load_2d(sa + C::A_BYTES, &tmW, &full_bar[stage], (kb0 + kb) * RF_BK, 0);
    issued |= 1u << stage;
    parity = (parity & ~(1u << stage)) | (phase << stage);
    if (++stage == a.stages) {
      stage = 0;
      phase ^= 1;
    }
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(tfull_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    // x may be the previous kernel's output
    pdl_wait();
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
    for (; kb_issued < nk && kb_issued < a.stages; ++kb_issued) issue(kb_issued);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_launch_dependents();

  if (warp >= 2) {
    // Warps 2..15 wait for the MMAs anyway: they run the routing step once on no token (every
    // slot invalid at run time, so it reads and writes nothing), which brings its code into
    // the instruction cache. The routing code runs only a few times per CTA, and fetching it
    // cold cost more than executing it.
    float v[NT][J];
    int t[NT];
    bool valid[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      t[n] = 0;
      valid[n] = a.T < 0;
#pragma unroll
      for (int j = 0; j < J; ++j) v[n][j] = static_cast<float>(lane + j);
    }
    RouteStats<J> none;
    none.zero();
    route_tokens<G, J, NT, FULL>(v, t, valid, a.T, a.E, a.k, a.gate_mode, a.select_bias,
                                 a.probs_t, a.topk_idx, a.topk_gate, none, err,
                                 SITE_ROUTE_NONFINITE);
  }

  if (warp == 0) {
    if (lane == 0 && nk > 0) {
      // ================= TMA producer: the rest of the K slice =================
      for (int kb = kb_issued; kb < nk; ++kb) {
        if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1, abort_flag, err,
                               SITE_GEMM_WAIT_EMPTY))
          break;
        issue(kb);
      }
      // every copy this thread issued has landed before the ring is reused or the CTA exits
      for (int s = 0; s < a.stages; ++s)
        if (issued & (1u << s))
          mbar_wait_bounded(&full_bar[s], (parity >> s) & 1u, nullptr, err, SITE_GEMM_WAIT_DRAIN);
    }
  } else if (warp == 1) {
    if (lane == 0 && nk > 0) {
      // ================= MMA issuer =================
      int mstage = 0;
      uint32_t mphase = 0;
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait_bounded(&full_bar[mstage], mphase, abort_flag, err, SITE_GEMM_WAIT_FULL))
          break;
        tc_fence_after();
        const uint32_t a_addr = smem_u32(ring + mstage * C::STAGE_BYTES);
        const uint32_t b_addr = a_addr + C::A_BYTES;
#pragma unroll
        for (int kk = 0; kk < RF_BK / 16; ++kk)
          tc_mma_bf16(tmem_base, smem_desc_kmajor<128>(a_addr + kk * 32),
                      smem_desc_kmajor<128>(b_addr + kk * 32), C::IDESC,
                      (kb | kk) != 0 ? 1u : 0u);
        tc_commit(&empty_bar[mstage]);
        if (++mstage == a.stages) {
          mstage = 0;
          mphase ^= 1;
        }
      }
      // after the last MMA (or an abort): everything issued has completed
      tc_commit(tfull_bar);
    }
  }
  __syncwarp();

  // ---- drain TMEM into the shared-memory block of partial logits (all warps: warp w reads
  // TMEM lane quarter w % 4, columns chunks w / 4, w / 4 + 4, ... of 16)
  {
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    float* prow = part + r * C::PSTRIDE;
    bool ok = true;
    if (nk > 0) ok = mbar_wait_bounded(tfull_bar, 0, abort_flag, err, SITE_GEMM_WAIT_TMEM_FULL);
    tc_fence_after();
#pragma unroll 1
    for (int c = warp >> 2; c < BN / 16; c += RF_WARPS / 4) {
      uint32_t v[16];
      if (nk > 0 && ok) {
        tmem_ld_16cols(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + c * 16, v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0u;   // an empty K slice contributes zeros
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(prow + c * 16 + 4 * q) =
            make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
  }
  tc_fence_before();
  // every CTA's partial logits are written and visible to the cluster
  if (a.cs > 1) cluster_sync_all(); else __syncthreads();

  // ---- reduce the cluster's partials in rank order and route this CTA's rows: warp w takes
  // TPW consecutive rows per iteration (32 / G token groups of NT rows each)
  constexpr int TPW = (32 / G) * NT;
  const int g = lane & (G - 1);
  const int gi = lane / G;
  RouteStats<J> st;
  st.zero();
  const int r_begin = static_cast<int>(rank) * RF_BM / a.cs;
  const int r_end = static_cast<int>(rank + 1) * RF_BM / a.cs;
  for (int base = r_begin + warp * TPW; base < r_end && row0 + base < a.T;
       base += RF_WARPS * TPW) {
    float v[NT][J];
    int t[NT];
    bool valid[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const int r = base + gi * NT + n;
      t[n] = row0 + r;
      valid[n] = r < r_end && t[n] < a.T;
    }
    // the partial rows: rank 0's, then each further rank's added in order; every load of a
    // rank is issued before the sums that use it
    bool use[NT][J];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int j = 0; j < J; ++j) {
        use[n][j] = valid[n] && (FULL || g + G * j < a.E);
        v[n][j] = 0.f;
      }
    const int r0 = base + gi * NT;
    if (a.cs == 1) {
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int j = 0; j < J; ++j)
          if (use[n][j]) v[n][j] = part[(r0 + n) * C::PSTRIDE + g + G * j];
    } else {
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int j = 0; j < J; ++j)
          if (use[n][j]) v[n][j] = ld_cluster_f32(part + (r0 + n) * C::PSTRIDE + g + G * j, 0);
      if constexpr (NT * J <= 4) {
        // few values per lane (small E, where the clusters are widest): every rank's loads
        // go out before the first sum, so the ranks' latencies overlap
        float w[8][NT][J];
#pragma unroll
        for (int q = 1; q < 8; ++q)
#pragma unroll
          for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int j = 0; j < J; ++j)
              w[q][n][j] = (q < a.cs && use[n][j])
                               ? ld_cluster_f32(part + (r0 + n) * C::PSTRIDE + g + G * j, q)
                               : 0.f;
#pragma unroll
        for (int q = 1; q < 8; ++q)
#pragma unroll
          for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int j = 0; j < J; ++j)
              if (q < a.cs) v[n][j] += w[q][n][j];
      } else {
        for (int q = 1; q < a.cs; ++q) {
          float w[NT][J];
#pragma unroll
          for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int j = 0; j < J; ++j)
              w[n][j] =
                  use[n][j] ? ld_cluster_f32(part + (r0 + n) * C::PSTRIDE + g + G * j, q) : 0.f;
#pragma unroll
          for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int j = 0; j < J; ++j) v[n][j] += w[n][j];
        }
      }
    }
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int j = 0; j < J; ++j)
        if (use[n][j]) {
          const int e = g + G * j;
          if (a.bias != nullptr) v[n][j] += __ldg(a.bias + e);
          if (a.logits_out != nullptr) a.logits_out[static_cast<size_t>(t[n]) * a.E + e] = v[n][j];
        }
    route_tokens<G, J, NT, FULL>(v, t, valid, a.T, a.E, a.k, a.gate_mode, a.select_bias,
                                 a.probs_t, a.topk_idx, a.topk_gate, st, err,
                                 SITE_ROUTE_NONFINITE);
  }

  // per-CTA sums of p_{t,i} and lse^2: over the warp's groups, then over the warps in a fixed
  // order, expert-major
  route_stats_warp_sum<G, J>(st);
  if (lane < G) {
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int e = g + G * j;
      if (FULL || e < a.E) s_stat[warp * (a.E + 1) + e] = st.pacc[j];
    }
    if (lane == 0) s_stat[warp * (a.E + 1) + a.E] = st.lse2;
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= a.E; e += RF_THREADS) {
    float acc = 0.f;
    for (int w = 0; w < RF_WARPS; ++w) acc += s_stat[w * (a.E + 1) + e];
    a.partials[static_cast<size_t>(e) * gridDim.x + blockIdx.x] = acc;
  }

  tc_fence_before();
  // no CTA leaves while a peer may still read its shared memory
  if (a.cs > 1) cluster_sync_all(); else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

int pick_bn(int E) {
  if (E <= 16) return 16;
  if (E <= 32) return 32;
  if (E <= 64) return 64;
  if (E <= 128) return 128;
  return 256;
}

template <int BN, int G, int J, int NT, bool FULL>
int launch_rf(const RouterFusedPlan& pl, const RfArgs& a, const void* x, const void* wr,
              cudaStream_t stream) {
  using C = RfCfg<BN>;
  if (!get_encoder()) return MOE_ERR_CUDA;
  CUtensorMap mX{}, mW{};
  if (!encode_2d(&mX, x, a.d, a.T, RF_BM, RF_BK)) return MOE_ERR_CUDA;
  if (!encode_2d(&mW, wr, a.d, a.E, BN, RF_BK)) return MOE_ERR_CUDA;
  auto kernel = router_fused_kernel<BN, G, J, NT, FULL>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  static std::once_flag once[64];
  static bool attr_ok[64];
  std::call_once(once[dev], [&]() {
    attr_ok[dev] = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        C::smem_bytes(C::max_stages(), 256)) == cudaSuccess;
  });
  if (a.stages > C::max_stages() || a.E > 256) return MOE_ERR_INVALID;
  if (!attr_ok[dev]) return MOE_ERR_CUDA;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(pl.cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(pl.grid));
  cfg.blockDim = dim3(RF_THREADS);
  cfg.dynamicSmemBytes = static_cast<size_t>(C::smem_bytes(a.stages, a.E));
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, kernel, mX, mW, a) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

template <int BN, int G, int J, int NT>
int launch_rf_gj(const RouterFusedPlan& pl, const RfArgs& a, const void* x, const void* wr,
                 cudaStream_t stream) {
  if (a.E == G * J) return launch_rf<BN, G, J, NT, true>(pl, a, x, wr, stream);
  return launch_rf<BN, G, J, NT, false>(pl, a, x, wr, stream);
}

}  // namespace

// Cluster size and ring depth, from the shape alone (148 is the B300 SM count), so the
// summation order of the partial logits -- and every bit of them -- depends on the shape
// only. One CTA per SM (clusters are placed one CTA per SM: cluster occupancy measured 74
// two-CTA and 15 eight-CTA clusters at once), the split of d doubling while the grid still
// fits in one wave.
RouterFusedPlan router_fused_plan(int T, int d, int E) {
  RouterFusedPlan pl{};
  const int tiles = (T + RF_BM - 1) / RF_BM;
  const int nk = (d + RF_BK - 1) / RF_BK;
  int cs = 1;
  while (cs < 8 && tiles * cs * 2 <= 148 && cs * 2 <= nk) cs *= 2;
  pl.cs = cs;
  pl.kb_per = (nk + cs - 1) / cs;
  pl.grid = tiles * cs;
  const int bn = pick_bn(E);
  const int stage = RF_BM * RF_BK * 2 + bn * RF_BK * 2;
  pl.stages = std::max(2, std::min({RF_MAX_STAGES, 192 * 1024 / stage, std::max(pl.kb_per, 2)}));
  return pl;
}

int launch_router_fused(const RouterFusedPlan& pl, const void* x, const void* w_router,
                        const RouteArgs& r, int d, cudaStream_t stream) {
  if (r.T == 0) return MOE_OK;
  if (r.E > 256) return MOE_ERR_UNSUPPORTED;
  if (pl.cs < 1 || pl.cs > 8 || (RF_BM % pl.cs) != 0) return MOE_ERR_INVALID;
  RfArgs a{};
  a.T = r.T;
  a.E = r.E;
  a.d = d;
  a.kb_per = pl.kb_per;
  a.stages = pl.stages;
  a.cs = pl.cs;
  a.bias = r.bias;
  a.select_bias = r.select_bias;
  a.logits_out = r.logits_out;
  a.probs_t = r.probs_t;
  a.k = r.k;
  a.gate_mode = r.gate_mode;
  a.topk_idx = r.topk_idx;
  a.topk_gate = r.topk_gate;
  a.partials = r.partials;
  a.err = r.err;
  const int bn = pick_bn(r.E);
#define MOE_RF_CASE(BN_, EMAX, G_, J_, NT_) \
  if (bn == BN_ && r.E <= EMAX) return launch_rf_gj<BN_, G_, J_, NT_>(pl, a, x, w_router, stream);
  MOE_RF_CASE(16, 8, 8, 1, 2)
  MOE_RF_CASE(16, 16, 8, 2, 2)
  MOE_RF_CASE(32, 32, 8, 4, 2)
  MOE_RF_CASE(64, 64, 8, 8, 1)
  MOE_RF_CASE(128, 128, 8, 16, 1)
  MOE_RF_CASE(256, 256, 16, 16, 1)
#undef MOE_RF_CASE
  return MOE_ERR_UNSUPPORTED;
}

}  // namespace moe
