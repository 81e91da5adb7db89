// Failure-path self-test: exercises the bounded-wait pattern that every pipeline wait in the
// tensor-core kernels uses, on a wait that nothing ever completes. No fault is involved: the
// wait gives up after its limit, records MOE_ERR_DEVICE_TIMEOUT in the status word, and the
// kernel returns normally.
#include "sm100_ptx.cuh"
#include "internal.h"

namespace moe {
namespace {

using namespace ptx;

// One thread waits on an mbarrier initialised for one arrival that never comes; when limit_ns
// has passed by %globaltimer it records the timeout and returns.
__global__ void k_selftest_bounded_wait(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(&bar, 0)) {
      if (globaltimer() - t0 > limit_ns) {
        record_error(status, MOE_ERR_DEVICE_TIMEOUT);
        break;
      }
    }
  }
}

}  // namespace

cudaError_t launch_selftest_bounded_wait(int* status, uint64_t limit_ns, cudaStream_t st) {
  k_selftest_bounded_wait<<<1, 32, 0, st>>>(status, (unsigned long long)limit_ns);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
