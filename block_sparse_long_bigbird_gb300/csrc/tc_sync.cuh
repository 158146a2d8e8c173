// Bounded waits shared by the tensor-core kernels: every mbarrier wait gives
// up after a time limit, records SA_ERR_TIMEOUT in the device status word and
// raises the CTA's abort flag, so no kernel can spin forever.
#pragma once

#include <stdint.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace sa {
namespace {  // internal linkage: every translation unit keeps its own copy
namespace tcsync {

constexpr uint32_t kSuspendNs = 100000;  // try_wait suspend hint

struct Ctl {
    volatile int *abort;
    unsigned *status;
    unsigned long long limit_ns;
};

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool try_wait_hint(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Per-thread wait, bounded in time: returns false (and leaves) once the CTA
// aborts. The first probe has no suspend hint (cheapest when the phase is
// already complete); later probes sleep in the hardware until the phase
// completes or the hint expires (the hint never exceeds the limit, so a short
// limit takes effect within about one limit). No warp-collective operation
// inside, so lanes of one warp may call it independently.
__device__ __forceinline__ bool wait_one(uint32_t bar, uint32_t parity, const Ctl &c) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const bool short_limit = c.limit_ns < kSuspendNs;
    const uint32_t hint = short_limit ? (uint32_t)c.limit_ns : kSuspendNs;
    // With the default limit the clock starts at the first hinted miss (no
    // timer read on the common path); a short limit starts it now.
    unsigned long long t0 = short_limit ? global_ns() : 0;
    while (!try_wait_hint(bar, parity, hint)) {
        if (*c.abort) return false;
        const unsigned long long now = global_ns();
        if (t0 == 0) {
            t0 = now;
        } else if (now - t0 > c.limit_ns) {
            *c.abort = 1;
            atomicOr(c.status, kDevTimeout);
            return false;
        }
    }
    return true;
}
// Warp-uniform wait: every lane probes the barrier itself (a divergent
// single-lane wait costs hundreds of cycles to reconverge), then one vote
// gives all lanes the same answer.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const Ctl &c) {
    const bool ok = wait_one(bar, parity, c);
    return __all_sync(0xffffffffu, ok);
}
// Drain wait: before a CTA frees its TMEM and exits, it waits for its own
// TMA copies and MMAs still in flight. It ignores the abort flag and has its
// own limit, independent of the pipeline waits' limit (SA_OPT_WAIT_LIMIT may
// be set very short): an asynchronous copy or MMA that was issued lands in
// microseconds, so one second only ends a drain whose phase never completes.
constexpr unsigned long long kDrainLimitNs = 1000000000ull;
__device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = global_ns();
    while (!ptx::mbar_try_wait(bar, parity))
        if (global_ns() - t0 > kDrainLimitNs) return;
}

}  // namespace tcsync
}  // namespace
}  // namespace sa
