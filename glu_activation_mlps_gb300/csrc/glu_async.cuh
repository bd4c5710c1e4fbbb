// Shared-memory barriers and bulk copies (cp.async.bulk) for the staged
// kernels.  Every wait is bounded by a clock budget of about a second: a wait
// that runs out returns false and the caller records it and stops, so no block
// can hang the GPU.
#pragma once
#include <cstdint>

namespace glu {

constexpr long long kWaitBudgetCycles = 2000000000LL;   // ~1 s at 2 GHz

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Waits for the phase with the given parity to complete; false if the clock
// budget ran out first.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity)
{
    const long long t0 = clock64();
    while (true) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
        if (clock64() - t0 > kWaitBudgetCycles) return false;
    }
}

// mbar_wait for long waits by many warps: each try_wait may suspend the
// thread until the phase completes (up to the hint, in nanoseconds), so a
// waiting warp takes no issue slots from the working ones.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity)
{
    const long long t0 = clock64();
    while (true) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity), "r"(1000000u)
            : "memory");
        if (done) return true;
        if (clock64() - t0 > kWaitBudgetCycles) return false;
    }
}

// Barrier `id` (1..15) over `count` threads (a multiple of 32) of the block.
__device__ __forceinline__ void named_barrier(int id, int count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// A 4-byte copy global -> shared (cp.async, cached at L1), for small pieces
// that the bulk copies cannot carry (unaligned, not a multiple of 16 bytes).
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// Makes the mbarrier's current phase wait also for this thread's cp.async
// copies issued so far: the pending arrival count goes up by one now and down
// by one when they have landed.
__device__ __forceinline__ void cp_async_arrive(uint32_t bar)
{
    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

}  // namespace glu
