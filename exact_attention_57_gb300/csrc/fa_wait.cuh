// fa_wait.cuh — the bounded mbarrier wait every warp role of the tensor-core
// kernels uses, so that no wait can spin forever.
#pragma once

#include "ptx.cuh"

namespace fa {

struct WaitCtl {
  volatile int *abort;            // the CTA's abort flag (shared memory)
  unsigned *status;               // the device status word
  unsigned long long limit_ns;    // give-up time for one wait
  unsigned role;                  // status bit of the waiting role
};

// Bounded wait for an mbarrier phase.  Returns false if the CTA is aborting
// (unless honour_abort is false) or the wait ran past the limit, in which case
// it raises the abort flag and records its role in the status word.
__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, const WaitCtl &w,
                                             bool honour_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 7u) == 0) {
      if (honour_abort && *w.abort) return false;
      if (globaltimer_ns() - t0 > w.limit_ns) {
        *w.abort = 1;
        atomicOr(w.status, w.role);
        return false;
      }
    }
  }
}

}  // namespace fa
