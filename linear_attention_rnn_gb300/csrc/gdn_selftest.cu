// gdn_selftest.cu -- self-test of the bounded waits every kernel here relies on.
//
// One block waits on an mbarrier that nothing ever signals.  The wait is the
// same bounded wait the walks, the preparation and the gradient kernels use for
// their TMA copies, MMAs and handshakes; it must give up after its limit, and
// the kernel must then record the timeout in the status word and return
// normally, so the context stays usable for the calls that follow.
#include "gdn_kernels.cuh"
#include "gdn_tc05.cuh"

namespace gdn {

namespace {

__global__ void k_selftest_wait(long long limit_cycles, int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::mbar_fence_init();
  }
  __syncthreads();
  const bool done = tc::mbar_wait(&bar, 0, limit_cycles);  // phase 0 never completes
  __syncthreads();
  if (threadIdx.x == 0) atomicOr(status, done ? 2 : 1);
}

}  // namespace

cudaError_t launch_selftest_wait(long long limit_ns, int* status, cudaStream_t s) {
  // the waits count SM cycles: convert at the device's maximum SM clock
  int dev = 0, khz = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev);
  if (e != cudaSuccess) return e;
  const long long cycles = limit_ns * (long long)khz / 1000000LL;
  k_selftest_wait<<<1, 32, 0, s>>>(cycles > 0 ? cycles : 1, status);
  return cudaGetLastError();
}

}  // namespace gdn
