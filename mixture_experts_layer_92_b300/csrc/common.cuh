// Shared device helpers for the MoE kernels: error word, bounded waits, bf16 packing,
// warp reductions, and the sm_100-family PTX wrappers (mbarrier, TMA, tcgen05).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "moe.h"  // include/ is on the include path

namespace moe {

// ------------------------------------------------------------------------------------
// Workspace header: the sticky error word and the location that set it.
// ------------------------------------------------------------------------------------
struct DeviceError {
  int code;       // first moe_status recorded (0 = none)
  int where;      // kernel/site id of the first error
  int detail;     // site-specific detail (e.g. offending index)
  unsigned done_count;  // statistics/loss kernel: finished column blocks (back to 0 after use)
  unsigned grid_count;  // grid barrier of the dispatch kernel: arrivals (back to 0 after use)
  unsigned grid_gen;    //                                     generation
};

enum ErrSite : int {
  SITE_ROUTE_NONFINITE = 1,
  SITE_DISPATCH_INDEX = 2,
  SITE_GEMM_WAIT_EMPTY = 10,
  SITE_GEMM_WAIT_FULL = 11,
  SITE_GEMM_WAIT_TMEM_FULL = 12,
  SITE_GEMM_WAIT_TMEM_EMPTY = 13,
  SITE_GEMM_WAIT_DRAIN = 14,
  SITE_DISPATCH_GRID_BARRIER = 20,
  SITE_F16_RANGE_X = 30,   // 8-bit-weight path: an activation outside fp16's finite range
  SITE_F16_RANGE_H = 31,   //                    an H value outside fp16's finite range
  SITE_MX_NONFINITE_X = 32, // block-scaled path: a non-finite activation in x
  SITE_MX_NONFINITE_H = 33, //                    a non-finite hidden value H
  SITE_SELFTEST_WAIT = 40, // moe_selftest_wait_timeout: a wait that nothing completes
};

__device__ __forceinline__ void record_error(DeviceError* e, int code, int where, int detail) {
  if (e == nullptr) return;
  if (atomicCAS(&e->code, 0, code) == 0) {
    e->where = where;
    e->detail = detail;
  }
}

// Upper bound of every spin-wait on the device, in nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------------------------
// Numeric helpers
// ------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Codes 2P and 2P+1 of four E4M3 codes (low byte first) -> their two values as fp16 (code
// 2P in the low half), with the hardware conversion (one instruction per pair; every finite
// E4M3 value, subnormals included, is exact in fp16). The two E4M3 NaN codes give NaN (this
// path expects finite codes).
template <int P>
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t four_codes) {
  const uint16_t two = static_cast<uint16_t>(P == 0 ? (four_codes & 0xffffu) : (four_codes >> 16));
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(two));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Largest finite fp16 value.
constexpr float kF16Max = 65504.0f;

// Dynamic shared memory one CTA may opt in to on sm_100-class GPUs (227 KB).
constexpr int kMaxDynSmem = 227 * 1024;

// Orders this thread's generic-proxy shared-memory writes before later async-proxy reads
// (tensor-core operand fetches) of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// silu with CUDA's fast exponential and fast division, for results rounded to bf16:
// z / (1 + e^-z); for very negative z, e^-z = inf and the quotient is 0.
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// Programmatic dependent launch. A kernel launched with the programmatic-serialization
// attribute may start while the previous kernel in the stream is still running: pdl_wait()
// blocks until the kernels it depends on have completed and their writes are visible (it
// returns at once for an ordinary launch), and pdl_launch_dependents() lets the next such
// kernel start launching. Every kernel launched through launch_pdl calls pdl_wait() before
// it reads anything an earlier kernel wrote.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------------------------
// mbarrier
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// CLUSTER: acquire at cluster scope (the phase may have been completed by arrivals from the
// peer CTA of a cluster), else at CTA scope.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  if constexpr (CLUSTER) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar_addr), "r"(parity)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar_addr), "r"(parity)
        : "memory");
  }
  return ok != 0;
}

// Waits until the phase with the given parity of `bar` has completed. Gives up (returns
// false) when `*abort` becomes non-zero or after kWaitLimitNs; on a timeout it records
// MOE_ERR_TIMEOUT at `site` and raises `*abort` so that the other roles stop too.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort, DeviceError* err,
                                                  int site) {
  const uint32_t addr = smem_u32(bar);
  if (mbar_try_wait<CLUSTER>(addr, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait<CLUSTER>(addr, parity)) return true;
    if ((i & 63u) == 0) {
      if (abort != nullptr && *abort) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        record_error(err, MOE_ERR_TIMEOUT, site, 0);
        if (abort != nullptr) *abort = 1;
        return false;
      }
    }
  }
}

// ------------------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), tensor maps passed as __grid_constant__ kernel parameters
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* m, uint64_t* bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* m, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Prefetch of one box of a 3-D tensor map into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* m, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

// The same loads for a CTA pair: the copy lands in this CTA's shared memory and completes
// its bytes on the mbarrier at cluster address `bar_cluster` (mapa), which may be the
// peer CTA's.
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* m,
                                                 uint32_t bar_cluster, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(void* smem_dst, const CUtensorMap* m,
                                                 uint32_t bar_cluster, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// Cluster (shared::cluster) address of the object at `p`'s offset in the cluster's CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}

// Tensor store shared -> global of one box (bulk-group completion; clipped at the tensor's
// bounds). The source must have been written before a fence_proxy_async_smem().
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, const void* smem_src, int c0,
                                             int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(smem_u32(smem_src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// One warp's 32-row block for a tensor store: row `lane`'s ROW_BYTES bytes (the 16-byte
// units words[4q .. 4q+3]) written into `buf` where a tensor map with ROW_BYTES-wide rows
// and the matching swizzle (128-, 64- or 32-byte) expects them: unit q of row r at q ^ (r % 8),
// q ^ (r / 2 % 4) or q ^ (r / 4 % 2). Every eight consecutive lanes then cover all 32 banks.
template <int ROW_BYTES>
__device__ __forceinline__ void stage_row_swizzled(uint8_t* buf, const uint32_t* words, int lane) {
  static_assert(ROW_BYTES == 128 || ROW_BYTES == 64 || ROW_BYTES == 32, "swizzle span");
#pragma unroll
  for (int q = 0; q < ROW_BYTES / 16; ++q) {
    const int pos = ROW_BYTES == 128 ? (q ^ (lane & 7))
                    : ROW_BYTES == 64 ? (q ^ ((lane >> 1) & 3))
                                      : (q ^ ((lane >> 2) & 1));
    *reinterpret_cast<uint4*>(buf + lane * ROW_BYTES + (pos << 4)) =
        make_uint4(words[4 * q], words[4 * q + 1], words[4 * q + 2], words[4 * q + 3]);
  }
}
// After every lane has staged its row: make the block visible to the async proxy and let
// lane 0 write it with one tensor store at (c0, c1) of `map` (one bulk group).
__device__ __forceinline__ void store_staged_2d(const CUtensorMap* map, const uint8_t* buf,
                                                int c0, int c1, int lane) {
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(buf)), "r"(c0), "r"(c1)
        : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  }
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until the issuing thread's bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// ... all but the most recent bulk group (double-buffered staging).
__device__ __forceinline__ void bulk_wait_group_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Wait until the issuing thread's bulk stores are complete.
__device__ __forceinline__ void bulk_wait_group0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ------------------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores, accumulators in tensor memory)
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Whole warp: allocate `ncols` TMEM columns; the base address is written to *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA with a 128- or
// 64-byte swizzle: rows of SW bytes, 8-row groups 8*SW bytes apart. Advancing along K inside
// a row is a plain start-address offset (the swizzle is applied to the absolute address).
template <int SW>
__device__ __forceinline__ uint64_t smem_desc_kmajor(uint32_t saddr) {
  static_assert(SW == 128 || SW == 64, "128- or 64-byte swizzle");
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address, 16-byte units
  d |= static_cast<uint64_t>(1) << 16;                    // leading byte offset (unused)
  d |= static_cast<uint64_t>((8 * SW) >> 4) << 32;        // stride byte offset: 8 rows
  d |= static_cast<uint64_t>(1) << 46;                    // descriptor version
  d |= static_cast<uint64_t>(SW == 128 ? 2 : 4) << 61;    // swizzle mode
  return d;
}

// Instruction descriptor, kind::f16 with bf16 A/B (both K-major) and fp32 accumulate.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4)                                   // D format: f32
         | (1u << 7)                                 // A format: bf16
         | (1u << 10)                                // B format: bf16
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// The same with fp16 A/B (format code 0): both operands of one MMA are fp16.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4)                                   // D format: f32
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// Shared-memory matrix descriptor for an MN-major operand tile written by TMA with a 128-byte
// swizzle as 64-element-wide chunks (boxes of [64 K rows, 64 M/N elements]): inside a chunk
// K row k sits at k*128 bytes and 8-row groups are 1024 bytes apart (stride byte offset);
// the chunks lie `chunk_bytes` apart along M/N (leading byte offset). Advancing K by 16 is
// a start-address offset of 2048 bytes.
__device__ __forceinline__ uint64_t smem_desc_mn_sw128(uint32_t saddr, uint32_t chunk_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);            // start address
  d |= static_cast<uint64_t>((chunk_bytes >> 4) & 0x3FFFu) << 16;  // leading byte offset
  d |= static_cast<uint64_t>(1024 >> 4) << 32;                     // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                             // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                             // 128-byte swizzle
  return d;
}

// Operand major-ness bits of the kind::f16 instruction descriptor: A (bit 15) and B (bit 16)
// read MN-major instead of K-major.
__host__ __device__ constexpr uint32_t idesc_major(bool a_mn, bool b_mn) {
  return (a_mn ? 1u << 15 : 0u) | (b_mn ? 1u << 16 : 0u);
}

__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------------------------------
// CTA pairs (thread-block clusters of two CTAs on two SMs; tcgen05 with cta_group::2).
// A kernel that uses these uses cta_group::2 for every tcgen05 alloc / mma / commit.
// ------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Every thread of both CTAs: arrive (release) and wait (acquire) on the cluster barrier.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// Arrive (release at cluster scope) on the mbarrier at the same shared-memory offset as `bar`
// in the cluster's CTA `rank` (which may be this CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint64_t* bar, uint32_t rank) {
  asm volatile(
      "{\n\t.reg .b32 ra;\n\t"
      "mapa.shared::cluster.u32 ra, %0, %1;\n\t"
      "mbarrier.arrive.release.cluster.shared::cluster.b64 _, [ra];\n\t}" ::"r"(smem_u32(bar)),
      "r"(rank)
      : "memory");
}

// One warp of EACH CTA of the pair: allocate `ncols` TMEM columns in both CTAs.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// One thread of the pair's leader CTA: D (M = 256 rows, half in each CTA's TMEM) += A . B^T,
// A's rows 0..127 and B's rows 0..N/2-1 read from this CTA's shared memory at the
// descriptors' addresses, the other halves from the same addresses in the peer CTA.
__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the mbarrier at `bar`'s offset in every CTA of `cta_mask` when all tcgen05
// operations issued so far by this thread are done.
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// ------------------------------------------------------------------------------------
// Block-scaled MMA (kind::mxf8f6f4): 8-bit (or 4-bit, unpacked to one byte in shared
// memory) operands with one UE8M0 scale per 32 K values, scales in tensor memory.
// ------------------------------------------------------------------------------------
// One contiguous copy global -> shared of `bytes` (multiple of 16, both addresses 16-byte
// aligned), completing on `bar`.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory descriptor of a contiguous [rows x 16 bytes] block without swizzle (8-row
// core matrices 128 bytes apart): the source of a scale-factor copy into tensor memory.
__device__ __forceinline__ uint64_t smem_desc_plain16(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address, 16-byte units
  d |= static_cast<uint64_t>(1) << 16;                    // leading byte offset (one column)
  d |= static_cast<uint64_t>(128 >> 4) << 32;             // stride byte offset: 8 rows
  d |= static_cast<uint64_t>(1) << 46;                    // descriptor version
  return d;
}

// One thread: copy a 512-byte scale atom (32 rows x 16 bytes) into 4 TMEM columns at
// `taddr`, replicated into all four 32-lane quarters.
__device__ __forceinline__ void tc_cp_scale_atom(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// Instruction descriptor of kind::mxf8f6f4 with UE8M0 scales: A E4M3 (format 0), B E4M3 (0)
// or E2M1 (5), both K-major; `sf` selects the byte of each scale column (K block of 32
// inside a 128-wide scale atom) for A (bits 29-30) and B (bits 4-5).
__host__ __device__ constexpr uint32_t idesc_mx(int M, int N, int b_format, int sf) {
  return (static_cast<uint32_t>(sf) << 4)           // B scale factor id
         | (static_cast<uint32_t>(b_format) << 10)  // B format (A format 0: E4M3)
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (1u << 23)                               // UE8M0 scales
         | (static_cast<uint32_t>(M >> 4) << 24)    // M / 16
         | (static_cast<uint32_t>(sf) << 29);       // A scale factor id
}

// D (M x N fp32 in TMEM) (+)= (A * scale_A) . (B * scale_B)^T over K = 32.
__device__ __forceinline__ void tc_mma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// 32 lanes x 32 columns of 32-bit accumulators: thread i gets row (lane base + i).
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_16cols(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

}  // namespace moe
