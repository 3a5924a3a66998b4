// waits.cuh -- bounded waits on mbarrier phases, shared by every pipelined kernel.
//
// No wait in this library can spin forever: after `timeout_ns` of global time it records
// MOE_ERR_TIMEOUT in the caller's status word, raises the CTA's abort flag so the other roles stop
// issuing work, and returns false. The caller then drains what it issued and returns.
#pragma once

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {

constexpr uint64_t kWaitTimeoutNs = 2000000000ull;   // 2 s: far beyond any legitimate wait

// Returns true once the phase with `parity` has completed; false if the CTA is aborting or the
// wait expired.
// kCluster: the phase may be completed by arrivals from another CTA of the cluster.
template <bool kCluster = false>
__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity) {
    return kCluster ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
}

template <bool kCluster = false>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           int* status, uint64_t timeout_ns = kWaitTimeoutNs) {
    if (try_wait<kCluster>(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (try_wait<kCluster>(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > timeout_ns) {
            *abort_flag = 1;
            set_status(status, MOE_ERR_TIMEOUT);
            return false;
        }
    }
}

// Wait used while draining after an abort: bounded, ignores the abort flag.
template <bool kCluster = false>
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity,
                                           uint64_t timeout_ns = kWaitTimeoutNs) {
    const uint64_t t0 = globaltimer_ns();
    while (!try_wait<kCluster>(bar, parity))
        if (globaltimer_ns() - t0 > timeout_ns) return;
}

}  // namespace moe
