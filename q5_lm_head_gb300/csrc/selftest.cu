// Self-test of the failure path every pipelined kernel relies on: a bounded
// mbarrier wait that gives up, records the timeout in the status word and lets
// the kernel return normally (no trap, no fault, the context stays usable).
#include "internal.h"
#include "ptx.cuh"

namespace muse {
namespace {

// One thread waits on an mbarrier that nothing ever arrives on.
__global__ void wait_timeout_selftest_kernel(uint32_t *status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !ptx::mbar_wait(&bar, 0)) atomicOr(status, kStatusWaitTimeout);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(uint32_t *status, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(status);
  return cudaGetLastError();
}

}  // namespace muse
