// Bulk copies between global and shared memory (the Blackwell TMA unit,
// 1-D cp.async.bulk) and the mbarrier that their loads complete on.  Every
// global address and size must be a multiple of 16 bytes; shared-memory
// destinations too.
#pragma once

#include <cstdint>

namespace dpz {

// About two seconds of SM clock: the bound on every wait for a bulk copy.
constexpr long long kWaitLimitCycles = 4000000000LL;

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

// Wait for phase 0 of the barrier, at most kWaitLimitCycles; false if the
// wait ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar)
{
    if (mbar_try_wait(bar, 0)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, 0))
        if (clock64() - t0 > kWaitLimitCycles) return false;
    return true;
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
