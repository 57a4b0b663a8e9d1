// zq_pair_wait.cuh -- bounded waits for the kernels that run as a CTA pair.
// A wait gives up after kWaitLimitNs; the CTA that gives up raises the
// device status bit, sets its own abort flag and the peer's (so every role of
// both CTAs stops at its next wait), and the roles then leave through the
// pair's teardown.  Each translation unit that includes this gets its own
// copies of the shared-memory flag and status pointer, which thread 0 of the
// kernel sets up.
#pragma once

#include <stdint.h>

#include "zq_async.cuh"
#include "zq_cluster.cuh"

namespace zq {
namespace {

// Bounded wait on a barrier that may receive arrivals from the peer CTA;
// gives up at once when either CTA of the pair has already failed.  Inline
// throughout: a call out of a warpgroup whose register count was changed
// would force spills around it.
// The pair's abort flag and the device status word live in shared memory
// (set up by thread 0), so a wait keeps only the peer's flag address in
// registers.
__shared__ int s_abort;
__shared__ unsigned int *s_status;

struct PairCtx {
    uint32_t abort_peer;   // cluster address of the peer's flag
};

__device__ __forceinline__ bool pair_wait(uint64_t *bar, uint32_t parity, const PairCtx &c)
{
    if (mbar_try_wait_cl(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    volatile int *abort_flag = &s_abort;
    for (;;) {
        if (*abort_flag) return false;
        if (mbar_try_wait_cl_sleep(bar, parity, kSleepNs)) return true;
        if (global_ns() - t0 >= kWaitLimitNs) {
            flag_timeout(s_status);
            *abort_flag = 1;
            st_cluster_u32(c.abort_peer, 1u);
            return false;
        }
    }
}

// The whole warp waits (every lane observes the phase itself, one warp-wide
// probe per try) and agrees on the outcome.  A lane-0 wait followed by a
// shuffle and __syncwarp cost more: the chunk kernel's converter, metadata
// and epilogue warps wait several times per super-block, and its [gate;up]
// launch at B = 8 took 50.0 us that way against 45.4 us.
__device__ __forceinline__ bool pair_warp_wait(uint64_t *bar, uint32_t parity, const PairCtx &c)
{
    return __all_sync(0xffffffffu, pair_wait(bar, parity, c));
}

// Latency-critical waits: up to 2000 non-suspending probes first, then the
// sleeping bounded wait.
__device__ __forceinline__ bool mbar_test_wait_cl(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool pair_wait_spin(uint64_t *bar, uint32_t parity, const PairCtx &c)
{
    for (int i = 0; i < 2000; ++i)
        if (mbar_test_wait_cl(bar, parity)) return true;
    return pair_wait(bar, parity, c);
}

__device__ __forceinline__ bool pair_lane0_wait_spin(uint64_t *bar, uint32_t parity, const PairCtx &c)
{
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = pair_wait_spin(bar, parity, c);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    __syncwarp();
    return ok;
}

// Bounded wait that ignores the abort flags (draining work already issued).
__device__ __forceinline__ bool drain_wait(uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait_cl_sleep(bar, parity, kSleepNs)) return true;
        if (global_ns() - t0 >= kWaitLimitNs) return false;
    }
}

__device__ __forceinline__ PairCtx pair_ctx(uint32_t rank)
{
    PairCtx c;
    c.abort_peer = cluster_addr(smem_u32(&s_abort), rank ^ 1u);
    return c;
}

}  // namespace
}  // namespace zq
