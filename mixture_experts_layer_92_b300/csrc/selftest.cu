// Diagnostic kernel for the library's failure path: one device wait on an mbarrier that
// nothing ever completes. It is the bounded wait every pipeline kernel uses (common.cuh):
// after its time limit it records MOE_ERR_TIMEOUT (site SITE_SELFTEST_WAIT) in the workspace
// error word and returns, so the GPU is neither trapped nor hung and the context stays
// usable. It lets a test check, on a real GPU, what a pipeline stall would report.
#include "common.cuh"
#include "launchers.h"

namespace moe {

namespace {

__global__ void wait_timeout_kernel(DeviceError* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);   // one arrival expected; none comes
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    mbar_wait_bounded(&bar, 0, reinterpret_cast<volatile int*>(&abort_flag), err,
                      SITE_SELFTEST_WAIT);
}

}  // namespace

int launch_wait_timeout(DeviceError* err, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(err);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
