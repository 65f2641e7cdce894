// A kernel whose bounded wait runs out on purpose, so that a test can check
// the failure detection every other kernel relies on: the wait gives up after
// its limit, records the timeout in the device status word and returns, and
// the context stays usable. Nothing else in the library calls it.

#include <cstdint>

#include "apr_internal.h"
#include "dev_common.cuh"

namespace apr {
namespace {

// One thread waits on an mbarrier that nothing ever arrives on, through the
// same bounded wait as the library's kernels, with the given limit.
__global__ void bounded_wait_kernel(unsigned long long limit_ns, unsigned* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_for(&bar, 0, &abort_flag, status, limit_ns);
}

}  // namespace

cudaError_t launch_bounded_wait(unsigned long long limit_ns, unsigned* status, cudaStream_t s) {
  bounded_wait_kernel<<<1, 32, 0, s>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace apr
