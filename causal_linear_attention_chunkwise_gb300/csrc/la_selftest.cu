// la_selftest.cu -- exercises the bounded-wait timeout path without faulting:
// one CTA waits on an mbarrier that nothing ever arrives at, gives up after
// `spin_limit` polls, records the timeout in the device error word and exits
// normally, leaving the context usable.
#include "la_common.cuh"
#include "la_internal.h"
#include "la_ptx.cuh"

namespace la {
namespace {

__global__ void wait_timeout_kernel(uint32_t spin_limit, unsigned int *err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // expects one arrival that never comes
    fence_mbarrier_init();
  }
  __syncthreads();
  bool done = mbar_wait_bounded(&bar, 0, spin_limit);
  if (!done && threadIdx.x == 0) record_device_error(err, KID_SELFTEST, 1);
  __syncthreads();
  if (threadIdx.x == 0) mbar_inval(&bar);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(unsigned int spin_limit, cudaStream_t s) {
  unsigned int *err = device_error_word();
  if (!err) return cudaErrorInvalidDevice;
  wait_timeout_kernel<<<1, 32, 0, s>>>(spin_limit, err);
  return cudaGetLastError();
}

}  // namespace la
