// moe_route_topk_noalloc: gates and top-k from precomputed logits without any workspace.
//
// Some callers cannot hand this library device memory: code that runs inside a host
// framework which owns every device allocation and forbids cudaMalloc (allocation
// synchronises the device and can stall other work), or a call site that has no allocator
// at hand. For them this entry point keeps its only scratch -- the per-block partial sums
// of the router statistics -- in a fixed-size array in the library's own device memory.
//
// The array is file-scope `static __device__` storage: every GPU that loads the library
// holds kNoAllocScratchBytes of it until the process exits, and every call on a device uses
// the same array. Calls that overlap on the GPU (for instance on two streams at once) race
// on it; serialise them. The kernels write every partial before reading it, so nothing has
// to be cleared between calls.
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "launchers.h"

namespace moe {
namespace {

// 2 MiB: partials of (E + 1) x route_blocks(T) floats (expert-major: the statistics of
// expert e for every block, then expert e + 1). Enough for any T when E <= 884 (at most 592
// blocks), and for larger E while T is small enough.
constexpr size_t kNoAllocScratchBytes = 2u << 20;

static __device__ __align__(256) float g_route_scratch[kNoAllocScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::once_flag g_setup_once[kMaxDevices];
float* g_scratch_ptr[kMaxDevices];
cudaError_t g_setup_status[kMaxDevices];

// Host code cannot use g_route_scratch as an address (it names a host-side stand-in); the
// device address is looked up once per device, with that device current.
cudaError_t scratch_for_current_device(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(g_setup_once[dev], [dev]() {
    void* p = nullptr;
    g_setup_status[dev] = cudaGetSymbolAddress(&p, g_route_scratch);
    g_scratch_ptr[dev] = static_cast<float*>(p);
  });
  if (g_setup_status[dev] != cudaSuccess) return g_setup_status[dev];
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

extern "C" int moe_route_topk_noalloc(const moe_shape* s, const float* logits_in,
                                      int32_t* topk_idx, float* topk_gate, float* stats,
                                      void* stream) {
  using namespace moe;
  const int rc = moe_check_shape(s);
  if (rc != MOE_OK) return rc;
  if (s->gate == MOE_GATE_EXPERT_CHOICE)
    return set_error_detail(MOE_ERR_UNSUPPORTED,
                            "expert-choice layers route with moe_expert_choice");
  // every pointer is checked before anything is queued, as the workspace entry points do
  auto misaligned4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) != 0; };
  if (stats != nullptr && misaligned4(stats))
    return set_error_detail(MOE_ERR_INVALID, "stats is not 4-byte aligned");
  if (s->T > 0) {
    if (logits_in == nullptr || topk_idx == nullptr || topk_gate == nullptr)
      return set_error_detail(MOE_ERR_INVALID, "logits_in, topk_idx and topk_gate are required");
    if (misaligned4(logits_in) || misaligned4(topk_idx) || misaligned4(topk_gate))
      return set_error_detail(MOE_ERR_INVALID,
                              "logits_in, topk_idx and topk_gate must be 4-byte aligned");
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (s->T == 0) {
    if (stats != nullptr && cudaMemsetAsync(stats, 0, (s->E + 1) * sizeof(float), st) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  const size_t need = static_cast<size_t>(route_blocks(s->T)) * (s->E + 1) * sizeof(float);
  if (need > kNoAllocScratchBytes) {
    char msg[160];
    snprintf(msg, sizeof(msg),
             "needs %zu bytes of scratch for T = %d, E = %d; the built-in scratch holds %zu",
             need, s->T, s->E, kNoAllocScratchBytes);
    return set_error_detail(MOE_ERR_UNSUPPORTED, msg);
  }
  float* partials = nullptr;
  const cudaError_t se = scratch_for_current_device(&partials);
  if (se != cudaSuccess) return set_error_detail(MOE_ERR_CUDA, cudaGetErrorString(se));
  RouteArgs a{};
  a.logits = logits_in;
  a.nsplit = 1;
  a.T = s->T;
  a.E = s->E;
  a.k = s->k;
  a.gate_mode = s->gate;
  a.topk_idx = topk_idx;
  a.topk_gate = topk_gate;
  a.partials = partials;
  int r = launch_route_topk(a, st);
  if (r != MOE_OK) return set_error_detail(r, "gates/top-k launch failed");
  if (stats != nullptr) r = launch_stats_reduce(partials, route_blocks(s->T), s->E, stats, st);
  if (r != MOE_OK) return set_error_detail(r, "statistics launch failed");
  return set_error_detail(MOE_OK, "");
}
