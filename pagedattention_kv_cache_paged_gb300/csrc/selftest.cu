// Self-test of the bounded waits every pipelined kernel relies on (the library's own failure path;
// nothing on the pages corresponds to it).
//
// One CTA of two warps.  Warp 0 waits on an mbarrier whose phase nothing completes, with the given
// limit, gives up and records PA_DEVERR_TIMEOUT and the launch's epoch in the device error word
// pair, exactly as a kernel whose TMA copy never lands would.  Warp 1 waits on a second such
// barrier with the kernels' own limit and must leave early once it sees its launch's epoch (the
// cooperative abort between waiting warps and CTAs of one launch).  Lane 0 of each warp stores how long its wait took.  No fault, trap or endless loop is
// involved: both waits end by themselves and the CUDA context stays usable.
#include "pa_common.cuh"
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {

__global__ void __launch_bounds__(64) selftest_wait_kernel(unsigned* err, unsigned epoch, uint64_t limit_ns,
                                                           unsigned long long* elapsed_ns) {
  __shared__ uint64_t bars[2];
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_barrier_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t t0 = globaltimer_ns();
  bool ok = true;
  if (lane == 0) ok = mbar_wait_for(&bars[warp], 0, err, epoch, warp == 0 ? limit_ns : kWaitLimitNs);
  const uint64_t t1 = globaltimer_ns();
  if (lane == 0) {
    if (!ok && warp == 0) raise_timeout(err, epoch);
    if (elapsed_ns != nullptr) elapsed_ns[warp] = t1 - t0;
  }
}

cudaError_t launch_selftest_wait(unsigned* err, unsigned epoch, uint64_t limit_ns, unsigned long long* elapsed_ns,
                                 cudaStream_t s, int* launches) {
  selftest_wait_kernel<<<1, 64, 0, s>>>(err, epoch, limit_ns, elapsed_ns);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace pa
