// Device helpers shared by the decode and prefill kernels.
#pragma once

#include <cstdint>

#include "gqa_common.h"
#include "ptx.cuh"

namespace gqa {

// Sequence lengths are clamped to [0, Tmax] on the device.
__device__ __forceinline__ int clamp_len(int t, int Tmax) { return t < 0 ? 0 : (t > Tmax ? Tmax : t); }

// Bounded wait on an mbarrier phase. On expiry, or when another warp of the
// CTA has already given up, it records the failure and returns false.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           unsigned* status, uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > timeout_ns) {
            *abort_flag = 1;
            atomicOr(status, kStatusTimeout);
            return false;
        }
    }
}

// Lane 0 waits (bounded) and the warp agrees on the outcome.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned* status, uint64_t timeout_ns) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = wait_phase(bar, parity, abort_flag, status, timeout_ns);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

}  // namespace gqa
