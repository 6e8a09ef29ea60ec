// cp_hold.cuh -- failure injection for the self-tests of the tf32 and backward
// kernels: a bounded wait on a flag that nothing sets.
#pragma once
#include <cstdint>

#include "cp_ptx.cuh"

namespace cpattn {

// Failure injection (self-tests only): wait, bounded by timeout_ns, for *hold
// to become non-zero.  A flag that nothing sets makes the wait run out; it then
// raises *abort_flag like any other bounded wait and returns false.
__device__ __forceinline__ bool hold_wait(const int *hold, uint64_t timeout_ns, volatile int *abort_flag) {
    const uint64_t t0 = global_timer_ns();
    while (*reinterpret_cast<const volatile int *>(hold) == 0) {
        if (global_timer_ns() - t0 > timeout_ns) {
            *abort_flag = 1;
            return false;
        }
        __nanosleep(1000);
    }
    return true;
}

}  // namespace cpattn
