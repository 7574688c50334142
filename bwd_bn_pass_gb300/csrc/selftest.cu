// Self-test of the bounded waits that every ring and flag wait of the
// library uses: a wait that nothing satisfies must give up after its limit,
// record GBN_DEV_WAIT_TIMEOUT in the device status word and return, leaving
// the context usable.  The kernel waits on an mbarrier whose one expected
// arrival never comes (no copy is in flight), through the same helper as the
// ring kernels.  Failure detection is thus exercised without faulting,
// trapping or hanging the GPU.
#include "gbn_common.cuh"
#include "gbn_internal.h"

namespace gbn {

namespace {

__global__ void bounded_wait_selftest_kernel(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  const bool done = mbar_wait_bounded(&bar, 0, limit_ns);
  if (!done && threadIdx.x == 0) report_status(status, GBN_DEV_WAIT_TIMEOUT);
}

}  // namespace

cudaError_t selftest_bounded_wait(int* status, uint64_t limit_ns, cudaStream_t st) {
  return launch(bounded_wait_selftest_kernel, dim3(1), dim3(32), 0, st, false, status, limit_ns);
}

}  // namespace gbn
