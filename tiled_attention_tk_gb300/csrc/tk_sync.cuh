// tk_sync.cuh -- bounded waits and the device status word shared by the
// kernels of one translation unit.  Every mbarrier wait in the library goes
// through wait_bounded: it gives up after a time limit, records
// TK_ERR_DEVICE_TIMEOUT (and where) in the status word, and raises the CTA's
// abort flag so that the other roles stop too.  Nothing traps or spins
// forever.  Each translation unit has its own status word (file-scope
// `static __device__`); the C ABI reads and clears all of them.
#pragma once

#include <cstdint>

#include "tk_attn.h"
#include "tk_ptx.cuh"

namespace tk {

static __device__ unsigned int g_status;  // 0 or TK_ERR_DEVICE_TIMEOUT
static __device__ unsigned int g_detail;  // where the first wait gave up

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far above any legitimate wait
constexpr uint64_t kDrainLimitNs = 50000000ull;   // 50 ms for draining after an abort

// Role tags of the `where` word: (role << 24) | (barrier << 16) | step.
enum : uint32_t {
    ROLE_PRODUCER = 1,
    ROLE_MMA = 2,
    ROLE_SOFTMAX = 3,
    ROLE_SELFTEST = 4,
    ROLE_BWD_PRODUCER = 5,
    ROLE_BWD_MMA = 6,
    ROLE_BWD_COMPUTE = 7,
    ROLE_BWD_LAYOUT = 8,  // not a wait: the backward kernel found its shared memory misaligned
    ROLE_EPILOGUE = 9,
    ROLE_LAYOUT = 10      // not a wait: the forward kernel found its shared memory misaligned
};

__device__ __forceinline__ void record_timeout(uint32_t where) {
    if (atomicCAS(&g_status, 0u, (unsigned)TK_ERR_DEVICE_TIMEOUT) == 0u) atomicExch(&g_detail, where);
}

// Waits for the phase `parity` of `bar`.  Returns false (and raises the
// CTA's abort flag) if the wait exceeds `limit_ns`, or if another thread of
// the CTA has raised the abort flag.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                             uint32_t where, uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((spin & 63u) == 0u) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > limit_ns || spin > 0x7FFFFFF0u) {
                *abort_flag = 1;
                record_timeout(where);
                return false;
            }
        }
    }
}

// One arrival per warp: the warp's lanes first synchronise (ordering their
// earlier writes, and after a tcgen05 fence their TMEM stores), then lane 0
// arrives.  Barriers fed this way count 4 arrivals per warpgroup.
__device__ __forceinline__ void warp_arrive(uint32_t bar, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

}  // namespace tk
