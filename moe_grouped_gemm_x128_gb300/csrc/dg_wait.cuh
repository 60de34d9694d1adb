// Bounded mbarrier waits shared by the library's kernels.  A wait gives up
// after a number of SM cycles, raises the CTA's abort flag and the
// DG_DEVFLAG_TIMEOUT bit of the device status word, and returns false, so
// that every role of the kernel can stop, let its asynchronous work drain and
// exit; nothing spins forever.
#pragma once

#include "dg_common.h"
#include "dg_ptx.cuh"

namespace dg {

// Pipeline waits give up after this many SM cycles (about 2 s at 2 GHz).
constexpr long long kWaitTimeoutCycles = 4000000000ll;

__device__ __forceinline__ void raise_status(unsigned int *status, unsigned int bit)
{
    atomicOr(status, bit);
}

// Slow path of wait_phase: poll until the phase completes, another role
// aborts, or about `limit` SM cycles pass.  The clock and the abort flag are
// looked at every 64 polls only: a timer read costs far more than a barrier
// test.
__device__ __forceinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                             unsigned int *status, long long limit)
{
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (mbar_test_wait(bar, parity))
            return true;
        if ((it & 63u) == 0) {
            if (*abort_flag)
                return false;
            if (clock64() - t0 > limit) {
                *abort_flag = 1;
                raise_status(status, DG_DEVFLAG_TIMEOUT);
                return false;
            }
        }
    }
}

// Bounded wait for the phase of `bar` with the given parity, by one thread:
// one inline test, then the polling loop.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                           unsigned int *status, long long limit = kWaitTimeoutCycles)
{
    if (mbar_test_wait(bar, parity))
        return true;
    return wait_phase_slow(bar, parity, abort_flag, status, limit);
}

// Bounded wait for the phase of `bar`, by a whole warp that stays converged:
// every lane tests, and the warp leaves together once every lane has seen the
// phase complete (the lanes then reach warp-wide instructions such as
// tcgen05.ld without reconverging).  Same limit and abort rule as
// wait_phase; returns the same value in every lane.
__device__ __forceinline__ bool wait_phase_warp(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                                unsigned int *status, long long limit = kWaitTimeoutCycles)
{
    if (__all_sync(0xffffffffu, mbar_test_wait(bar, parity)))
        return true;
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (__all_sync(0xffffffffu, mbar_test_wait(bar, parity)))
            return true;
        if ((it & 63u) == 0) {
            const bool aborted = *abort_flag != 0;
            const bool late = clock64() - t0 > limit;
            if (__any_sync(0xffffffffu, aborted || late)) {
                if (__any_sync(0xffffffffu, late && !aborted) && (threadIdx.x & 31) == 0) {
                    *abort_flag = 1;
                    raise_status(status, DG_DEVFLAG_TIMEOUT);
                }
                return false;
            }
        }
    }
}

// Bounded wait used while shutting down after an abort (ignores the flag).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, long long limit = kWaitTimeoutCycles)
{
    const long long t0 = clock64();
    for (uint32_t it = 1; !mbar_test_wait(bar, parity); ++it)
        if ((it & 63u) == 0 && clock64() - t0 > limit)
            return;
}

}  // namespace dg
