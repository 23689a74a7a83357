// Self-test of the bounded device-side wait used by the decode pipeline.
//
// One CTA initialises an mbarrier that nothing will ever arrive on and waits
// for it with the same bounded wait the decode kernels use (mbar_wait_bounded).
// The wait must give up after `limit_ns`, record MT_STATUS_BIT_TIMEOUT in the
// caller's status word and return, leaving the CUDA context usable. Nothing
// here faults, traps or hangs: the wait is bounded by time and by poll count.
#include "common.cuh"
#include "internal.h"

namespace mtkv {
namespace {

__global__ void bounded_wait_selftest_kernel(unsigned long long limit_ns, uint32_t *status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait_bounded(&bar, 0, &abort_flag, limit_ns)) report(status, MT_STATUS_BIT_TIMEOUT);
    // complete the pending phase so the barrier is quiescent before exit
    mbar_arrive(&bar);
  }
}

}  // namespace
}  // namespace mtkv

using namespace mtkv;

extern "C" mt_status mt_selftest_bounded_wait(uint64_t limit_ns, uint32_t *status,
                                              mt_stream stream) {
  if (!status) return fail(MT_ERR_INVALID_ARG, "mt_selftest_bounded_wait: null status word");
  if (limit_ns == 0 || limit_ns > 2000000000ull)
    return fail(MT_ERR_INVALID_ARG, "mt_selftest_bounded_wait: limit must be in (0, 2 s]");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  bounded_wait_selftest_kernel<<<1, 32, 0, s>>>((unsigned long long)limit_ns, status);
  mt_status st = cuda_check(cudaGetLastError(), "mt_selftest_bounded_wait launch");
  return st == MT_OK ? ok() : st;
}
