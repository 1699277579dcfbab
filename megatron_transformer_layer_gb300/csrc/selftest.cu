// Self-tests of the failure paths the library's kernels rely on: a bounded
// mbarrier wait that runs out records MC_ERR_DEVICE_TIMEOUT and where in the
// status word, and the kernel returns, leaving the context usable; an index
// check that fails (the check of a debug build's stores) records
// MC_ERR_DEVICE_BOUNDS and skips the access.
#include <cuda_runtime.h>

#include "mc_layer_internal.h"
#include "ptx.cuh"

namespace mc {
namespace {

// One warp waits (bounded) on an mbarrier that nothing arrives on.
__global__ void wait_timeout_kernel(uint64_t timeout_ns, int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait_warp_limit(&bar, 0, status, kSiteSelfTest, timeout_ns);
}

// Writes 1 to buf[index] only if the index check against `extent` passes.
__global__ void bounds_check_kernel(int64_t index, int64_t extent, int* buf, int* status) {
  if (check_index(index >= 0 && index < extent, status, kSiteSelfTest)) buf[index] = 1;
}

}  // namespace
}  // namespace mc

using namespace mc;

extern "C" int mc_selftest_bounds_check(int64_t index, int64_t extent, int* buf, int* status,
                                        void* stream) {
  if (!status || !buf) return MC_ERR_NULLPTR;
  if (extent < 1) return MC_ERR_ARGUMENT;
  bounds_check_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(index, extent, buf, status);
  return cudaGetLastError() == cudaSuccess ? MC_OK : MC_ERR_CUDA;
}

extern "C" int mc_selftest_wait_timeout(int64_t timeout_ns, int* status, void* stream) {
  if (timeout_ns < 1000 || timeout_ns > 100000000) return MC_ERR_ARGUMENT;  // 1 us .. 100 ms
  if (!status) return MC_ERR_NULLPTR;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint64_t>(timeout_ns), status);
  return cudaGetLastError() == cudaSuccess ? MC_OK : MC_ERR_CUDA;
}
