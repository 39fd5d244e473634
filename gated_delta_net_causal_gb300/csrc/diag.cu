// gdn_selftest_wait_timeout: a bounded device-side wait made to run out on
// purpose, so that the give-up path (status word, clean kernel exit, usable
// context) can be checked on the device without any fault or hang. One warp
// waits on an mbarrier that nothing arrives on; no copy or MMA is in flight.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(uint64_t limit_ns, int32_t* gave_up) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_abort;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival expected; none ever comes
    s_abort = 0;
    fence_mbar_init();
  }
  __syncwarp();
  const bool done = mbar_wait_bounded(&bar, 0, &s_abort, limit_ns);
  if (threadIdx.x == 0) *gave_up = done ? 0 : 1;
}

}  // namespace

cudaError_t launch_wait_timeout(uint64_t limit_ns, int32_t* gave_up, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns, gave_up);
  return cudaGetLastError();
}

}  // namespace gdn

GDN_DEFINE_ERROR_READER(diag)
