// Self-test of the library's failure handling: the bounded waits.
//
// Every wait of the pipelined kernels (on an mbarrier phase, or on a global
// completion counter another CTA raises) gives up after a time limit, records
// MOE_ERR_TIMEOUT in the workspace's status word and lets the kernel leave
// cleanly, so a lost signal ends as an error code the host reads, never as a
// hung GPU. This kernel exercises exactly those two wait helpers on a barrier
// that nothing arms and a counter that nothing raises, with a short limit, so
// a test can observe the expiry without stalling any real kernel.
#include "tc_common.cuh"

namespace moe {
namespace {

using namespace tc;

// result[0] = 1 if the barrier wait succeeded (it must not), result[1] the
// same for the counter wait; result[2], result[3] = the time each wait took
// before giving up, in microseconds.
__global__ void wait_expiry_kernel(int32_t *status, const int32_t *counter, unsigned long long limit_ns,
                                   int32_t *result) {
  __shared__ unsigned long long bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival completes phase 0; none ever comes
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    abort_flag = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile int *abort = &abort_flag;
    unsigned long long t0 = globaltimer();
    const bool a = mbar_wait(&bar, 0u, abort, status, kKSelfTest, 1, limit_ns);
    const unsigned long long t1 = globaltimer();
    *abort = 0;  // the barrier wait raised it; the counter wait runs its own limit
    const bool b = wait_counter(counter, 1, abort, status, kKSelfTest, 2, limit_ns);
    const unsigned long long t2 = globaltimer();
    result[0] = a ? 1 : 0;
    result[1] = b ? 1 : 0;
    result[2] = (int32_t)((t1 - t0) / 1000ull);
    result[3] = (int32_t)((t2 - t1) / 1000ull);
  }
}

}  // namespace

cudaError_t launch_wait_expiry(int32_t *status, const int32_t *counter, unsigned long long limit_ns,
                               int32_t *result, cudaStream_t s) {
  wait_expiry_kernel<<<1, 32, 0, s>>>(status, counter, limit_ns, result);
  return cudaGetLastError();
}

}  // namespace moe
