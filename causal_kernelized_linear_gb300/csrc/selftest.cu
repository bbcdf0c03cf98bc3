// Self-tests of the failure paths: la_selftest_wait_timeout (one CTA waits,
// with the waits of the tensor-core kernels, on an mbarrier that nothing
// signals, and must give up with LA_ERR_TIMEOUT in the status word) and
// la_selftest_device_check (a device-side check of the LA_DEBUG build that
// fails and must record LA_ERR_DEVICE_CHECK without making the access).
#include "common.cuh"
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

// One thread guards an access with an index one past a 4-element buffer.  In
// an LA_DEBUG build the check fails, records LA_ERR_DEVICE_CHECK with site 90
// and the access is skipped; the index is masked as well, so the access stays
// inside the buffer in any build.
__global__ void __launch_bounds__(32, 1) selftest_check_kernel(int* status, int i, int* sink) {
  __shared__ int buf[4];
  if (threadIdx.x == 0) {
    buf[0] = buf[1] = buf[2] = buf[3] = 0;
    if (LA_DCHECK(status, i >= 0 && i < 4, 90)) buf[i & 3] = 1;
    if (sink) *sink = buf[0] + buf[1] + buf[2] + buf[3];
  }
}

}  // namespace

cudaError_t selftest_check(int* status, cudaStream_t stream) {
  selftest_check_kernel<<<1, 32, 0, stream>>>(status, 4, nullptr);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t selftest_wait(int* status, uint64_t limit_ns, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 64, 0, stream>>>(status, limit_ns);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace la
