// Bulk-copy staging variant of the streaming kernels, for contiguous operands.
//
// One or two blocks per SM (see BulkShape).  Warp 0 is the producer: one lane moves fixed-size chunks
// of every input operand from global into a ring of shared-memory stages with
// cp.async.bulk (the Blackwell bulk-copy engine), completing on an mbarrier per
// stage.  Warps 1..kBulkConsumers consume: wait for a stage, read it from
// shared memory, compute exactly as the direct kernels do (same element ops),
// store the outputs straight to global memory with 16-byte stores, and release
// the stage.  The loads in flight per SM are the whole ring, independent of
// registers or occupancy.
//
// Every wait is bounded by a clock budget (about a second).  A wait that runs
// out adds one to a device counter the host can read, stops the block from
// issuing or consuming, waits (again bounded) for the copies it already
// issued, and returns, so no block can hang the GPU.
// Included by glu_bulk.cu only.
#pragma once
#include "glu_async.cuh"
#include "glu_internal.h"
#include "glu_kernels.cuh"

namespace glu {

constexpr int kBulkChunk = 16384;                       // bytes per operand per stage
static_assert(kBulkChunk == kBulkChunkHost, "host view of the bulk chunk");

// Two shapes: WIDE = one block per SM with 8 consumer warps and a 192 KiB
// ring; NARROW = two blocks per SM, each with 16 consumer warps and a 96 KiB
// ring (the same bytes in flight per SM, four times the consumer warps).
template <int DIR, bool NARROW>
struct BulkShape {
    static constexpr int kConsumers = NARROW ? 16 : 8;
    static constexpr int kThreads = 32 * (1 + kConsumers);
    static constexpr int kRingBudget = NARROW ? 98304 : 196608;
    static constexpr int kIn = DIR == kBwd ? 3 : 2;
    static constexpr int kOut = DIR == kBwd ? 2 : 1;
    static constexpr int kStages = kRingBudget / (kIn * kBulkChunk);
    static constexpr int kRingBytes = kStages * kIn * kBulkChunk;
    static constexpr int kSmemBytes = kRingBytes + 2 * kStages * 8 + 16;
    static_assert(kStages >= 2, "at least double buffering");
};

// Waits that ran out, summed over all bulk launches since the last reset.
static __device__ unsigned int g_bulk_timeouts;

template <class Act, class T, int DIR, bool NARROW>
__global__ void __launch_bounds__(BulkShape<DIR, NARROW>::kThreads, NARROW ? 2 : 1)
    glu_bulk_kernel(const BulkParams p)
{
    using S = BulkShape<DIR, NARROW>;
    constexpr int kBulkConsumers = S::kConsumers;
    using C = Codec<T>;
    constexpr bool kExact = std::is_same<T, float>::value;
    constexpr int PW = C::kPerWord;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::kRingBytes);
    uint64_t *empty = full + S::kStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + S::kStages);

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S::kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), kBulkConsumers);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const int64_t stride = gridDim.x;
    if (warp == 0) {
        if (lane != 0) return;
        const char *src[3] = {p.a, p.b, p.dc};
        int64_t issued = 0;
        for (int64_t it = 0;; ++it) {
            const int64_t c = blockIdx.x + it * stride;
            if (c >= p.chunks || *abort_flag) break;
            const int s = int(it % S::kStages);
            if (it >= S::kStages &&
                !mbar_wait(smem_u32(&empty[s]), uint32_t((it / S::kStages - 1) & 1))) {
                atomicAdd(&g_bulk_timeouts, 1u);
                *abort_flag = 1;
                break;
            }
            const uint32_t bar = smem_u32(&full[s]);
            mbar_expect_tx(bar, S::kIn * kBulkChunk);
            for (int op = 0; op < S::kIn; ++op) {
                const char *g = src[op] + c * kBulkChunk;
                bulk_load(smem_u32(ring + (size_t(s) * S::kIn + op) * kBulkChunk), g, kBulkChunk, bar);
            }
            issued = it + 1;
        }
        // The block may only exit once every copy it issued has landed.
        const int64_t first = issued > S::kStages ? issued - S::kStages : 0;
        for (int64_t it = first; it < issued; ++it)
            if (!mbar_wait(smem_u32(&full[it % S::kStages]), uint32_t((it / S::kStages) & 1))) {
                atomicAdd(&g_bulk_timeouts, 1u);
                break;
            }
        return;
    }

    // consumers
    const int ct = threadIdx.x - 32;                       // 0 .. 32 * kBulkConsumers - 1
    constexpr int kVecs = kBulkChunk / 16;                 // 16-byte vectors per operand per chunk
    constexpr int kPerThread = kVecs / (32 * kBulkConsumers);
    static_assert(kVecs % (32 * kBulkConsumers) == 0, "chunk must split evenly over consumers");
    for (int64_t it = 0;; ++it) {
        const int64_t c = blockIdx.x + it * stride;
        if (c >= p.chunks || *abort_flag) break;
        const int s = int(it % S::kStages);
        if (!mbar_wait(smem_u32(&full[s]), uint32_t((it / S::kStages) & 1))) {
            if (lane == 0) atomicAdd(&g_bulk_timeouts, 1u);
            *abort_flag = 1;
            break;
        }
        const unsigned char *st = ring + size_t(s) * S::kIn * kBulkChunk;
#pragma unroll
        for (int v = 0; v < kPerThread; ++v) {
            const int vi = v * 32 * kBulkConsumers + ct;
            uint4 va = *reinterpret_cast<const uint4 *>(st + 0 * kBulkChunk + vi * 16);
            uint4 vb = *reinterpret_cast<const uint4 *>(st + 1 * kBulkChunk + vi * 16);
            uint4 vc = make_uint4(0, 0, 0, 0);
            if constexpr (DIR == kBwd) vc = *reinterpret_cast<const uint4 *>(st + 2 * kBulkChunk + vi * 16);
            const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
            const uint32_t wc[4] = {vc.x, vc.y, vc.z, vc.w};
            uint32_t o0[4], o1[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float f0[PW], f1[PW];
                if constexpr (DIR == kFwd) fwd_word<Act, kExact, C>(wa[j], wb[j], f0);
                else bwd_word<Act, kExact, C>(wa[j], wb[j], wc[j], f0, f1);
                o0[j] = C::put(f0);
                if constexpr (DIR == kBwd) o1[j] = C::put(f1);
            }
            const int64_t off = c * kBulkChunk + int64_t(vi) * 16;
            Access<16>::store(p.y0 + off, o0);
            if constexpr (DIR == kBwd) Access<16>::store(p.y1 + off, o1);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    }
}

}  // namespace glu
