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

}  // namespace gqa
