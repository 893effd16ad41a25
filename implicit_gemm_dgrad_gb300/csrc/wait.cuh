// Bounded pipeline waits shared by the sm_103a kernels: every mbarrier wait
// gives up after the launch's wait limit (CDG_WAIT_LIMIT_NS unless the plan
// sets another), records CDG_ERR_TIMEOUT in the launch's status word and
// raises the CTA's abort flag, so that no wait can hang a GPU.
#pragma once

#include "cdg_params.h"
#include "ptx.cuh"

namespace cdg {

constexpr int kTimeoutStatus = 6;  // CDG_ERR_TIMEOUT

struct Ctl {
    volatile uint32_t *abort;
    int *status;
    uint64_t limit = CDG_WAIT_LIMIT_NS;  // nanoseconds a single wait may take
};

// Slow path of a pipeline wait: spin on try_wait (which itself suspends the
// thread for a while) until the phase completes, the CTA aborts, or the wait
// runs past ctl.limit, in which case it records the timeout.
static __device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, Ctl ctl)
{
    const uint64_t t0 = global_timer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 15u) == 0) {
            if (*ctl.abort) return false;
            if (global_timer_ns() - t0 > ctl.limit) {
                *ctl.abort = 1u;
                atomicCAS(ctl.status, 0, kTimeoutStatus);
                return false;
            }
        }
    }
}

// Wait for phase `parity` of barrier `bar`; false if the CTA is aborting.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, Ctl ctl)
{
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, ctl);
}

}  // namespace cdg
