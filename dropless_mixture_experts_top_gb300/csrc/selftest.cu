// selftest.cu -- a diagnostic that exercises the bounded pipeline wait.
//
// Every mbarrier wait in the library's kernels is bounded (mbar_wait): after
// about two seconds of SM clock it gives up, the kernel drains its own work,
// sets MOE_DEV_WAIT_TIMEOUT in the call's status word and returns, so a lost
// arrival shows up as a status the host can read instead of a hung GPU.  This
// kernel waits on an mbarrier that nothing arrives at, through the same
// mbar_wait, to show that path end to end without faulting or hanging.
#include <cuda_runtime.h>

#include "../../include/moe.h"
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(int32_t *status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival expected; none ever comes
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  int ok = 1;
  if (threadIdx.x == 0) ok = mbar_wait(&bar, 0, &abort_flag) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (threadIdx.x == 0 && !ok) flag_status(status, kDevWaitTimeout);
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_selftest_wait_timeout(int32_t *device_status, void *stream) {
  if (!device_status) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(device_status) & 3u) return MOE_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(device_status, 0, sizeof(int32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
  moe::wait_timeout_kernel<<<1, 32, 0, s>>>(device_status);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
