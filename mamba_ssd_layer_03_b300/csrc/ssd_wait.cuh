// Bounded device-side waits shared by the fused kernel and the library's
// self-test of its failure path.  Every wait gives up after kWaitLimitNs of
// wall-clock time (%globaltimer), records SSD_ERR_DEVICE_TIMEOUT in the call's
// status word and returns false, so that a kernel whose partner never arrives
// still finishes and leaves the context usable.
#pragma once

#include <stdint.h>

#include "../../include/ssd.h"
#include "ssd_device.cuh"
#include "tc_ptx.cuh"

namespace ssd {
namespace wait {

using namespace tc;

__device__ __forceinline__ int ld_acquire_i(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_i(int *p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// mbarrier.try_wait with a suspend-time hint: a waiting thread sleeps (and
// issues nothing) until the phase completes or about `ns` have passed.
__device__ __forceinline__ bool try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// Bounded wait.  Once it has waited far longer than any healthy step takes
// (20 us), it also gives up as soon as the call's status word records an
// error, so that a failed call finishes quickly; the status word is not read
// before then because that global read would delay the wake-up.
__device__ __forceinline__ bool fwait(uint64_t *bar, uint32_t parity, int *status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        // not unrolled: every wait site inlines this loop, and the kernels'
        // instruction footprint matters more than the loop's few branches
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (try_wait_sleep(bar, parity, 2000)) return true;
        const uint64_t dt = globaltimer_ns() - t0;
        if (dt > 20000ull && status_bad(status)) return false;
        if (dt > kWaitLimitNs) {
            set_status(status, SSD_ERR_DEVICE_TIMEOUT);
            return false;
        }
    }
}

// Bounded wait for a flag in global memory that another CTA sets with a
// release store (the state handed over at a lane split).  Also gives up as
// soon as the status word records an error.
__device__ __forceinline__ void wait_flag(const int *flag, int *status) {
    const uint64_t tw = globaltimer_ns();
    while (ld_acquire_i(flag) == 0) {
        if (status_bad(status)) break;
        if (globaltimer_ns() - tw > kWaitLimitNs) {
            set_status(status, SSD_ERR_DEVICE_TIMEOUT);
            break;
        }
        __nanosleep(64);
    }
}

}  // namespace wait
}  // namespace ssd
