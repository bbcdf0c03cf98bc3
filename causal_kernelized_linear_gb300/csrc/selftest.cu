// Self-test of the bounded-wait failure path (la_selftest_wait_timeout): one
// CTA waits, with the waits of the tensor-core kernels, on an mbarrier that
// nothing signals, and must give up with LA_ERR_TIMEOUT in the status word.
#include "internal.h"
#include "tc.cuh"

namespace la {
namespace {

using namespace tc;

// Warp 0: the whole-warp wait (every lane polls, the warp agrees on the
// outcome).  Warp 1, lane 0: the single-thread wait of the producer and MMA
// roles, entered after the abort flag is set, so it must return at once.
__global__ void __launch_bounds__(64, 1) selftest_wait_kernel(int* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int abort_flag;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);   // one arrival completes the phase; none ever comes
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (warp == 0) warp_wait(&bar, 0, status, &abort_flag, limit_ns);
  __syncthreads();
  if (warp == 1 && (threadIdx.x & 31) == 0) mbar_wait(&bar, 0, status, &abort_flag, limit_ns);
}

}  // namespace

cudaError_t selftest_wait(int* status, uint64_t limit_ns, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 64, 0, stream>>>(status, limit_ns);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace la
