// pa_selftest.cu -- exercises the kernels' bounded-wait failure path on the
// device without a fault: a wait on an mbarrier that nothing arrives on must
// give up after its limit, record PA_STATUS_TIMEOUT and return, leaving the
// context usable.  The wait routines used here (mbar_wait_for and its
// warp-uniform form) are the ones behind every pipeline barrier of the
// attention kernels, which call them with the 2 s limit kWaitLimitNs.
#include "pa_launch.cuh"

namespace pa {
namespace {

__global__ void __launch_bounds__(64, 1) wait_selftest_kernel(uint64_t limit_ns, int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival expected; none is ever made
    fence_mbar_init();
  }
  __syncthreads();
  bool ok = false;
  if (threadIdx.x < 32) {
    // warp 0: the warp-uniform wait taken before tensor-memory operations
    ok = mbar_wait_warp_for(&bar, 0, status, limit_ns);
  } else if (threadIdx.x == 32) {
    // warp 1, one thread: the single-thread wait of the producer and MMA roles
    ok = mbar_wait_for(&bar, 0, status, limit_ns);
  }
  // a wait that reported success on a phase nobody completed would be a bug:
  // flag it with a second bit so the host can tell the two outcomes apart
  if (__syncthreads_or(ok) && threadIdx.x == 0 && status) atomicOr(status, PA_STATUS_BAD_LENGTH);
}

}  // namespace

cudaError_t launch_wait_selftest(uint64_t limit_ns, int32_t* status, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 64, 0, stream>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace pa
