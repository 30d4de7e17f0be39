// k_selftest.cu - a check of the bounded waits every kernel of the library relies on.
//
// Each wait of a kernel on an mbarrier (a page copy landing, a slot freed, an MMA done) gives up after a bounded
// time, records bit 8 in the device error word and lets the kernel return, so that a lost arrival cannot hang the
// GPU. This kernel runs that same bounded wait on a barrier that nothing completes, with no copy and no MMA
// outstanding, so that the give-up path itself can be exercised without any fault.
#include "../../include/kap.h"
#include "kap_device.cuh"
#include "kap_launch.h"

namespace kap {
namespace {

__global__ void wait_probe_kernel(uint32_t polls, uint32_t suspend_ns, int *err, int32_t *timed_out) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival would complete phase 0; none comes
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) *timed_out = mbar_wait_bounded(&bar, 0u, err, polls, suspend_ns) ? 0 : 1;
  __syncthreads();
  if (threadIdx.x == 0) mbar_inval(&bar);
}

}  // namespace

cudaError_t launch_wait_probe(uint32_t polls, uint32_t suspend_ns, int *err, int32_t *timed_out, cudaStream_t s) {
  wait_probe_kernel<<<1, 32, 0, s>>>(polls, suspend_ns, err, timed_out);
  return cudaGetLastError();
}

}  // namespace kap
