// Failure-detection self-test: one tiny kernel whose only wait can never be
// satisfied, so the library's bounded-wait rule (give up after a limit,
// record STATUS_TIMEOUT in the status word, return) is exercised on the GPU
// without a fault, a trap or a hang.  which = 0: an mbarrier phase that
// nothing completes (the helper every TMA wait uses); which = 1: a global
// word that nothing writes (the helper of the readiness polls).
#include "internal.h"

namespace {

__global__ void selftest_wait_kernel(DevStatus* st, const unsigned* never_set, int which, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  if (which == 0) {
    mbar_init(&bar, 1);   // expects one arrival that never comes
    fence_mbar_init();
    mbar_wait_limit(&bar, 0, st, limit);
  } else {
    flag_wait_limit(never_set, 1u, st, limit);
  }
}

}  // namespace

cudaError_t launch_selftest_wait(DevStatus* st, const unsigned* never_set, int which, long long limit,
                                 cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(st, never_set, which, limit);
  return cudaGetLastError();
}
