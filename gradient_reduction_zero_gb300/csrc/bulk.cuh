// Bulk copies between global and shared memory (the Blackwell TMA unit,
// 1-D cp.async.bulk) and the mbarrier that their loads complete on.  Every
// global address and size must be a multiple of 16 bytes; shared-memory
// destinations too.
#pragma once

#include <cstdint>

namespace dpz {

// About two seconds of SM clock: the bound on every wait for a bulk copy.
constexpr long long kWaitLimitCycles = 4000000000LL;

// How a staged kernel waits for its tile: the bound on each wait (SM clock
// cycles), and the bytes its barrier expects beyond the tile's loads.  That is
// 0 except in the self-test of the timeout path, where the barrier then never
// completes and the wait runs out (with a short bound, so the test is quick).
struct WaitSpec {
    long long limit;
    uint32_t extra_tx;
};
constexpr WaitSpec kWaitNormal{kWaitLimitCycles, 0u};

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Initialise a one-arrival mbarrier and make it visible to the copy engine.
__device__ __forceinline__ void mbar_init_one(uint64_t* bar)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive once and expect `bytes` of copies to complete on the barrier.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of the barrier with the given parity, at most `limit`
// SM clock cycles; false if the wait ran out.  The clock keeps counting while
// the context is switched out, so a wait that sees the limit pass polls once
// more before it gives up: a copy that completed while the context was off the
// GPU is then still taken.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, long long limit,
                                                  uint32_t parity = 0)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > limit) return mbar_try_wait(bar, parity);
    return true;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may begin once every block of the kernel before it on the
// stream has exited or called pdl_launch_dependents, before that kernel's
// writes are flushed; wait_prior blocks until every earlier kernel has
// completed and its writes are visible.  In a kernel launched the ordinary way
// it returns at once.
__device__ __forceinline__ void pdl_wait_prior()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next kernel on the stream, if it was launched with programmatic
// stream serialisation, be placed on the GPU now (it waits for this one with
// pdl_wait_prior before it touches memory).
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// The start of every kernel of this library: wait until the kernels before it
// on the stream have completed and their writes are visible, then let the
// next one be placed.  Nothing before this touches global memory, so a call
// launched early (programmatic stream serialisation) reads what the calls
// before it wrote, and back-to-back calls overlap one launch with the
// previous kernel's execution.
__device__ __forceinline__ void pdl_enter()
{
    pdl_wait_prior();
    pdl_launch_dependents();
}

// global -> shared, completing `bytes` on the mbarrier
__device__ __forceinline__ void bulk_load(void* sdst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(sdst)),
        "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// shared -> global, in the current bulk group
__device__ __forceinline__ void bulk_store(void* gdst, const void* ssrc, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_addr(ssrc)), "r"(bytes)
                 : "memory");
}

}  // namespace dpz
