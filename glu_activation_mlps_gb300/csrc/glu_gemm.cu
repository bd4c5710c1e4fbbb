// Gate and up projections with the gated activation in the epilogue, on the
// fifth-generation tensor cores of sm_103a:
//
//     y[m, i] = act(sum_k x[m, k] w_gate[i, k]) * (sum_k x[m, k] w_up[i, k])
//
// ("Skill: Write a Triton SiLU-Mul (SwiGLU) Kernel", Purpose and Performance
// requirements, "Versus epilogue fusion": the activation runs while the gate
// and up tiles are still on chip, so they never reach HBM; "Fused Kernels",
// section 4: gate and up tiles computed as x @ gate^T and x @ up^T.)
//
// A persistent grid walks tiles of y, BN columns wide.  Each block has three
// roles.  Warp 0 moves 64-wide K slices into a ring of shared-memory stages
// with the tensor-memory accelerator (128-byte swizzle).  One thread of warp 1
// issues tcgen05.mma (kind::f16, K = 16) into an fp32 [gate | up] accumulator
// of 2 BN tensor-memory columns per row; tensor memory holds two of them, so
// the MMAs of the next tile run while warps 2-5 read the finished one with
// tcgen05.ld (one row per thread), apply the same fp32 activation as the
// streaming kernels and round once.  Each warp stages 32 x 32 boxes of y in
// shared memory (64-byte swizzle) and the tensor-memory accelerator stores
// them, so y leaves in whole 128-byte lines; when y's rows are not 16-byte
// multiples the warps store from registers instead.
//
// Two shapes:
//   * one block per tile of 128 rows: the stage holds the x slice and the gate
//     and up slices back to back, and one MMA of N = 2 BN covers both;
//   * a cluster of two blocks per tile of 256 rows (cta_group::2): each block
//     loads its own 128 rows of x, block 0 the gate slice and block 1 the up
//     slice, and block 0 issues MMAs of M = 256, N = 2 BN that read the x rows
//     of both blocks and the gate and up halves of N from one block each; each
//     block's tensor memory receives [gate | up] for its own rows.  Every weight
//     byte crosses L2 -> shared memory once per 256 rows instead of once per 128.
// Tiles are ordered in groups of row blocks that share the weight slices in
// flight, so the weights stream from HBM about once.
//
// Every wait is bounded by a clock budget (about a second); a wait that runs
// out is counted in a device word (read by glu_wait_timeouts) and raises the
// abort flag of the block (and of its partner): every role leaves its loop, the
// copies and MMAs already issued are waited for (bounded), tensor memory is
// freed and the block returns with the remaining tiles unwritten.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "glu.h"
#include "glu_kernels.cuh"
#include "glu_internal.h"

namespace glu {
namespace gemm {

constexpr int BM = 128;                  // rows of x per block (tensor-memory lanes)
constexpr int BK = 64;                   // K per stage: 64 x 2 bytes = one 128-byte swizzle row
constexpr int kThreads = 192;            // warp 0 loads, warp 1 issues MMAs, warps 2-5 store
constexpr int kEpiWarps = 4;
constexpr int kRingBytes = 192 * 1024;   // shared memory given to the stage ring
constexpr int kYBox = 32;                // y leaves through 32 x 32 boxes (64-byte rows, 64-byte swizzle)
constexpr long long kBudget = 2000000000LL;   // ~1 s at 2 GHz

template <int BN, int CTAS>
struct Shape {
    static constexpr int kTileA = BM * BK * 2;
    static constexpr int kTileB = BN * BK * 2;                        // one of gate, up
    static constexpr int kStageBytes = kTileA + (CTAS == 1 ? 2 : 1) * kTileB;
    static constexpr int kStages = kRingBytes / kStageBytes > 8 ? 8 : kRingBytes / kStageBytes;
    static constexpr int kMmaM = BM * CTAS;
    static constexpr int kMmaN = 2 * BN;
    static constexpr int kAccCols = 2 * BN;                           // [gate | up] of one tile
    // two tiles in flight, in a power-of-two allocation
    static constexpr int kTmemCols = 2 * kAccCols <= 256 ? 256 : 512;
    static constexpr int kBars = 2 * kStages + 2 + 2 + 1;             // full, empty, acc_full, acc_empty, done
    static constexpr int kStageY = kEpiWarps * 2 * kYBox * kYBox * 2;  // two y boxes per epilogue warp
    static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kStageY + kBars * 8 + 16;
    static_assert(CTAS == 1 || CTAS == 2, "one block or a pair");
    static_assert(BN % 32 == 0 && BN >= 32 && kMmaN <= 256, "one MMA covers N = 2 BN <= 256");
    static_assert(2 * kAccCols <= kTmemCols, "two accumulators fit the allocation");
    static_assert(kTileA % 1024 == 0 && kTileB % 1024 == 0, "swizzle atoms stay 1024-byte aligned");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory per block");
};

struct Params {
    char *y;
    int64_t y_stride;       // bytes
    int M, I, K;
    int k_tiles;
    int m_blocks, i_blocks; // row blocks of 128 * CTAS rows, column blocks of BN
    int group_m;            // row blocks per group of the tile order
    int vec_store;          // y rows and base 16-byte aligned
    uint32_t a_bytes;       // bytes of x one block's copy brings per stage (rows that exist, up to 128)
    int tma_store;          // the same: y leaves through shared memory and the tensor-memory accelerator
};

static __device__ unsigned int g_gemm_timeouts;

__device__ __forceinline__ uint32_t saddr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Waits for the phase with the given parity to complete: spinning on
// try_wait, for the producer and MMA threads that must react at once; false
// once the clock budget has run out (checked every 16 tries).
__device__ __forceinline__ bool wait_parity(uint32_t bar, uint32_t parity)
{
    const long long t0 = clock64();
    for (uint32_t n = 1;; ++n) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
        if ((n & 15) == 0 && clock64() - t0 > kBudget) return false;
    }
}

// The same for the epilogue warps, which wait for a whole tile's MMAs: each
// try_wait may suspend the warp until the phase completes (200 us at most), so
// the waiting warps take no issue slots from the producer and MMA threads on
// their sub-partitions (measured 1-3 % faster than spinning).
__device__ __forceinline__ bool wait_parity_sleep(uint32_t bar, uint32_t parity)
{
    const long long t0 = clock64();
    while (true) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity), "r"(200000u)
            : "memory");
        if (done) return true;
        if (clock64() - t0 > kBudget) return false;
    }
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Shared::cluster address of the same shared variable in block `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void arrive_local(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void arrive_cluster(uint32_t bar_cluster)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

__device__ __forceinline__ void arrive_expect_tx_local(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Shared-memory matrix descriptor of a K-major tile stored as 128-byte rows
// with the 128-byte swizzle: start address, leading byte offset (unused for
// swizzled K-major tiles, encoded 1), stride byte offset 1024 (eight rows form
// one swizzle atom), the fixed version bits 0b001 at 46, swizzle mode 2 at 61.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr)
{
    uint64_t d = 0;
    d |= uint64_t((addr & 0x3FFFF) >> 4);
    d |= uint64_t(1) << 16;
    d |= uint64_t(1024 >> 4) << 32;
    d |= uint64_t(1) << 46;
    d |= uint64_t(2) << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator (bits
// 4-5 = 1), A and B formats (bits 7-9, 10-12: 0 = f16, 1 = bf16), both
// K-major (bits 15, 16 = 0), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f16(int ab_format, int M, int N)
{
    return (1u << 4) | (uint32_t(ab_format) << 7) | (uint32_t(ab_format) << 10) |
           (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// 2-D tiled copy into this block's shared memory; the barrier may belong to
// the partner block when CTAS == 2.
template <int CTAS>
__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar)
{
    if constexpr (CTAS == 1)
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
            "[%4];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
            : "memory");
    else
        asm volatile(
            "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
            "{%2, %3}], [%4];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
            : "memory");
}

template <int CTAS>
__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    if constexpr (CTAS == 1)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(acc)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(acc)
            : "memory");
}

// Arrive on `bar` (same offset in every block of the pair) once all MMAs this
// thread issued so far are done.
template <int CTAS>
__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    if constexpr (CTAS == 1)
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                     : "memory");
    else
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                bar),
            "h"(uint16_t(3))
            : "memory");
}

template <int CTAS>
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t cols)
{
    if constexpr (CTAS == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    } else {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
}

template <int CTAS>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols)
{
    if constexpr (CTAS == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}

// 32 consecutive fp32 columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// A 32 x 32 box of y from shared memory (64-byte swizzle) to global memory;
// the tensor-memory accelerator drops rows and columns outside y.
__device__ __forceinline__ void tma_store(const CUtensorMap *map, uint32_t src, int x, int y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

__device__ __forceinline__ void st_shared16(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// Tile t of the grouped order: group_m row blocks side by side walk the column blocks.
__device__ __forceinline__ void tile_origin(const Params &p, int t, int &mb, int &ib)
{
    const int per_group = p.group_m * p.i_blocks;
    const int first_m = (t / per_group) * p.group_m;
    const int gsize = min(p.m_blocks - first_m, p.group_m);
    const int r = t % per_group;
    mb = first_m + r % gsize;
    ib = r / gsize;
}

// The plain product D = A B^T (the down projection of an MLP) runs on the same
// kernel with PlainGemm in place of the activation: a tile is 2 BN output
// columns, the two weight slots hold consecutive BN-row slices of the one B
// matrix, and the epilogue only rounds the fp32 sums.
struct PlainGemm {};

// 32 fp32 accumulator columns of one row rounded once and packed two per word.
template <class Cd>
__device__ __forceinline__ void plain_pack(const uint32_t (&g)[32], uint32_t (&packed)[16])
{
    static_assert(Cd::kPerWord == 2, "16-bit outputs");
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const float f[2] = {__uint_as_float(g[j]), __uint_as_float(g[j + 1])};
        packed[j / 2] = Cd::put(f);
    }
}

// y = act(g) * u for 32 accumulator columns of one row, two at a time (the
// pair forms of the 16-bit path), rounded once and packed two per word.
template <class Act, class Cd>
__device__ __forceinline__ void epilogue_pack(const uint32_t (&g)[32], const uint32_t (&u)[32], uint32_t (&packed)[16])
{
    static_assert(Cd::kPerWord == 2, "16-bit outputs");
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const f2 gg = make_float2(__uint_as_float(g[j]), __uint_as_float(g[j + 1]));
        const f2 uu = make_float2(__uint_as_float(u[j]), __uint_as_float(u[j + 1]));
        const f2 y = mul2(Act::fwd2(gg), uu);
        const float f[2] = {y.x, y.y};
        packed[j / 2] = Cd::put(f);
    }
}

template <class Act, class T, int BN, int CTAS>
__global__ void __launch_bounds__(kThreads, 1)
    glu_gemm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_wg,
                    const __grid_constant__ CUtensorMap tm_wu, const __grid_constant__ CUtensorMap tm_y,
                    const Params p)
{
    using S = Shape<BN, CTAS>;
    using Cd = Codec<T>;
    constexpr int ST = S::kStages;
    constexpr bool kPlain = std::is_same<Act, PlainGemm>::value;
    constexpr int kOutCols = kPlain ? 2 * BN : BN;      // output columns of one tile
    constexpr uint32_t kIdesc = idesc_f16(std::is_same<T, __nv_bfloat16>::value ? 1 : 0, S::kMmaM, S::kMmaN);

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = saddr(smem_raw);
    unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);     // 1024-byte aligned ring
    unsigned char *ystage = smem + ST * S::kStageBytes;                     // 1024-byte aligned
    uint64_t *full = reinterpret_cast<uint64_t *>(ystage + S::kStageY);
    uint64_t *empty = full + ST;
    uint64_t *acc_full = empty + ST;            // [2]: MMAs of a tile done
    uint64_t *acc_empty = acc_full + 2;         // [2]: the epilogue (of both blocks) has read a tile
    uint64_t *done = acc_empty + 2;             // every MMA issued for this block, done
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(done + 1) + 1;

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = CTAS == 1 ? 0u : cluster_rank();     // block of the pair
    const int cluster = blockIdx.x / CTAS, n_clusters = gridDim.x / CTAS;
    const int n_tiles = p.m_blocks * p.i_blocks;

    // a timed-out wait stops this block and its partner
    auto raise_abort = [&]() {
        atomicAdd(&g_gemm_timeouts, 1u);
        *abort_flag = 1;
        if constexpr (CTAS == 2) {
            const uint32_t other = mapa(saddr(const_cast<int *>(abort_flag)), rank ^ 1u);
            asm volatile("st.relaxed.cluster.shared::cluster.u32 [%0], %1;" ::"r"(other), "r"(1) : "memory");
        }
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < ST; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&full[s])) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&empty[s])) : "memory");
        }
        for (int b = 0; b < 2; ++b) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&acc_full[b])) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(&acc_empty[b])),
                         "r"(kEpiWarps * CTAS)
                         : "memory");
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(done)) : "memory");
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) tmem_alloc<CTAS>(saddr(const_cast<uint32_t *>(tmem_slot)), S::kTmemCols);
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    if constexpr (CTAS == 2)
        cluster_sync();         // the partner's barriers are initialised before any copy signals them
    else
        __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == 0) {
        if (lane == 0) {
            // producer: stage s = it % ST is filled for the (it / ST)-th time
            uint32_t it = 0;
            for (int t = cluster; t < n_tiles && !*abort_flag; t += n_clusters) {
                int mb, ib;
                tile_origin(p, t, mb, ib);
                const int m0 = mb * S::kMmaM + int(rank) * BM, i0 = ib * kOutCols;
                const int i1 = kPlain ? i0 + BN : i0;          // rows of the second weight slot
                for (int kt = 0; kt < p.k_tiles; ++kt, ++it) {
                    const uint32_t s = it % ST, use = it / ST;
                    if (*abort_flag) break;
                    if (use > 0 && !wait_parity(saddr(&empty[s]), (use - 1) & 1)) {
                        raise_abort();
                        break;
                    }
                    const uint32_t st = saddr(smem + s * S::kStageBytes);
                    if constexpr (CTAS == 1) {
                        const uint32_t bar = saddr(&full[s]);
                        arrive_expect_tx_local(bar, p.a_bytes + uint32_t(2 * S::kTileB));
                        tma_load<1>(st, &tm_x, kt * BK, m0, bar);
                        tma_load<1>(st + S::kTileA, &tm_wg, kt * BK, i0, bar);
                        tma_load<1>(st + S::kTileA + S::kTileB, &tm_wu, kt * BK, i1, bar);
                    } else {
                        // both blocks' copies count on block 0's barrier, which
                        // alone arrives, expecting the bytes of the pair (block
                        // 1's copies may land first: the phase cannot complete
                        // before that arrival)
                        uint32_t bar = saddr(&full[s]);
                        if (rank == 0)
                            arrive_expect_tx_local(bar, uint32_t(2 * S::kStageBytes));
                        else
                            bar = mapa(bar, 0);
                        tma_load<2>(st, &tm_x, kt * BK, m0, bar);
                        tma_load<2>(st + S::kTileA, rank == 0 ? &tm_wg : &tm_wu, kt * BK, rank == 0 ? i0 : i1, bar);
                    }
                }
            }
            // block 0 holds the barriers of every copy of the pair: wait for the
            // last ones to land before the block may exit
            if (rank == 0) {
                const uint32_t first = it > uint32_t(ST) ? it - ST : 0;
                for (uint32_t j = first; j < it; ++j)
                    if (!wait_parity(saddr(&full[j % ST]), (j / ST) & 1)) {
                        atomicAdd(&g_gemm_timeouts, 1u);
                        break;
                    }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            if (rank == 0) {
                uint32_t it = 0;
                int lt = 0;
                for (int t = cluster; t < n_tiles; t += n_clusters, ++lt) {
                    if (*abort_flag) break;
                    const int ab = lt & 1, use_acc = lt >> 1;
                    if (use_acc > 0 && !wait_parity(saddr(&acc_empty[ab]), (use_acc - 1) & 1)) {
                        raise_abort();
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t d = tmem + uint32_t(ab * S::kAccCols);
                    bool ok = true;
                    for (int kt = 0; kt < p.k_tiles; ++kt, ++it) {
                        const uint32_t s = it % ST, use = it / ST;
                        if (!wait_parity(saddr(&full[s]), use & 1)) {
                            raise_abort();
                            ok = false;
                            break;
                        }
                        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                        const uint32_t a0 = saddr(smem + s * S::kStageBytes);
                        const uint64_t da = desc_sw128(a0);
                        const uint64_t db = desc_sw128(a0 + S::kTileA);
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk) {
                            // K advances by 16 elements = 32 bytes inside the swizzle row
                            const uint64_t step = uint64_t(kk * 32 >> 4);
                            mma<CTAS>(d, da + step, db + step, kIdesc, (kt | kk) != 0);
                        }
                        mma_commit<CTAS>(saddr(&empty[s]));     // the stage is free once these MMAs finish
                    }
                    if (!ok) break;
                    mma_commit<CTAS>(saddr(&acc_full[ab]));     // the tile's accumulator is complete
                }
                mma_commit<CTAS>(saddr(done));
            }
            // no MMA may still read this block's shared memory or write its tensor memory
            if (!wait_parity(saddr(done), 0)) atomicAdd(&g_gemm_timeouts, 1u);
        }
    } else {
        // epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. +31, one row per thread
        const int q = warp & 3;
        const uint32_t lane_base = uint32_t(q * 32) << 16;
        uint32_t n_boxes = 0;           // y boxes this warp has handed to the copy engine
        int lt = 0;
        for (int t = cluster; t < n_tiles; t += n_clusters, ++lt) {
            if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) break;
            const int ab = lt & 1, use_acc = lt >> 1;
            // tcgen05.ld is warp-collective: the whole warp takes one decision
            const bool ok = __all_sync(0xFFFFFFFFu, wait_parity_sleep(saddr(&acc_full[ab]), use_acc & 1));
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            if (!ok) {
                if (lane == 0) raise_abort();
                break;
            }
            int mb, ib;
            tile_origin(p, t, mb, ib);
            const int m = mb * S::kMmaM + int(rank) * BM + q * 32 + lane;
            const int i0 = ib * kOutCols;
            const uint32_t acc = tmem + lane_base + uint32_t(ab * S::kAccCols);
#pragma unroll 1
            for (int c0 = 0; c0 < kOutCols; c0 += 32) {
                uint32_t g[32], u[32];
                tmem_ld32(acc + uint32_t(c0), g);
                if constexpr (!kPlain) tmem_ld32(acc + uint32_t(BN + c0), u);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                if (c0 + 32 == kOutCols) {    // all of this tile read: hand the accumulator back
                    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (CTAS == 1)
                            arrive_local(saddr(&acc_empty[ab]));
                        else
                            arrive_cluster(mapa(saddr(&acc_empty[ab]), 0));
                    }
                }
                uint32_t packed[16];
                if constexpr (kPlain)
                    plain_pack<Cd>(g, packed);
                else
                    epilogue_pack<Act, Cd>(g, u, packed);
                if (p.tma_store) {
                    // this warp's 32 rows x 32 columns: row `lane` is 64 bytes,
                    // its 16-byte chunk c stored at chunk c ^ ((lane / 2) % 4)
                    const uint32_t buf = saddr(ystage) + uint32_t(q * 2 + (n_boxes & 1)) * (kYBox * kYBox * 2);
                    if (lane == 0 && n_boxes >= 2)      // the box stored from this buffer has been read
                        asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                    __syncwarp();
                    const uint32_t row = buf + uint32_t(lane) * 64u, sw = (uint32_t(lane) >> 1) & 3u;
#pragma unroll
                    for (uint32_t c = 0; c < 4; ++c)
                        st_shared16(row + ((c ^ sw) << 4), packed[4 * c], packed[4 * c + 1], packed[4 * c + 2],
                                    packed[4 * c + 3]);
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) tma_store(&tm_y, buf, i0 + c0, m - lane);
                    ++n_boxes;
                    continue;
                }
                if (m >= p.M) continue;
                const int i = i0 + c0;
                char *dst = p.y + int64_t(m) * p.y_stride + int64_t(i) * int64_t(sizeof(T));
                if (p.vec_store && i + 32 <= p.I) {
#pragma unroll
                    for (int v = 0; v < 32 / Cd::kPerWord / 4; ++v) {
                        const uint32_t w4[4] = {packed[4 * v], packed[4 * v + 1], packed[4 * v + 2],
                                                packed[4 * v + 3]};
                        Access<16>::store(dst + 16 * v, w4);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (i + j < p.I)
                            Cd::store1(dst + j * int64_t(sizeof(T)),
                                       Cd::get(packed[j / Cd::kPerWord], j % Cd::kPerWord));
                    }
                }
            }
        }
        // every box this warp stored has left shared memory and reached global memory
        if (lane == 0 && n_boxes > 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        __syncwarp();
    }

    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    if constexpr (CTAS == 2)
        cluster_sync();         // neither block leaves while the other may still signal its barriers
    else
        __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc<CTAS>(tmem, S::kTmemCols);
    }
}

}  // namespace gemm
}  // namespace glu

// ---------------------------------------------------------------- host side

namespace glu {
namespace gemm {
namespace {

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn()
{
    static std::once_flag once;
    static EncodeFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(p);
        else
            (void)cudaGetLastError();
    });
    return fn;
}

// A rows x cols row-major matrix (row stride in bytes) as a 2-D tensor map
// with a box of box_cols x box_rows; loads read zeros outside the matrix and
// stores drop what falls outside it.
bool make_map(CUtensorMap *m, bool bf16, const void *base, int64_t rows, int64_t cols, int64_t stride_bytes,
              int box_cols, int box_rows, CUtensorMapSwizzle swizzle)
{
    EncodeFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(stride_bytes)};
    const cuuint32_t box[2] = {cuuint32_t(box_cols), cuuint32_t(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

using KernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, Params);
constexpr int kPlainAct = 4;        // the kernel table's index of the plain product

template <class T, int BN, int CTAS>
KernelFn pick_act(int act)
{
    switch (act) {
    case 0: return glu_gemm_kernel<Silu, T, BN, CTAS>;
    case 1: return glu_gemm_kernel<GeluErf, T, BN, CTAS>;
    case 2: return glu_gemm_kernel<GeluTanh, T, BN, CTAS>;
    case 3: return glu_gemm_kernel<Relu, T, BN, CTAS>;
    case 4: return glu_gemm_kernel<PlainGemm, T, BN, CTAS>;     // D = A B^T
    default: return nullptr;
    }
}

struct Variant {
    KernelFn fn;
    int smem;
    int id;         // 0..5, see pick()
};

template <int BN, int CTAS>
Variant variant(bool bf16, int act, int id)
{
    return {bf16 ? pick_act<__nv_bfloat16, BN, CTAS>(act) : pick_act<__half, BN, CTAS>(act),
            Shape<BN, CTAS>::kSmemBytes, id};
}

Variant pick(bool bf16, int act, int bn, int ctas)
{
    if (ctas == 1) {
        if (bn == 64) return variant<64, 1>(bf16, act, 0);
        return bn == 96 ? variant<96, 1>(bf16, act, 1) : variant<128, 1>(bf16, act, 2);
    }
    if (bn == 64) return variant<64, 2>(bf16, act, 3);
    return bn == 96 ? variant<96, 2>(bf16, act, 4) : variant<128, 2>(bf16, act, 5);
}

// Column-tile width.  The kernel is bound by the stream of operand tiles into
// shared memory: a tile BN columns wide moves a_rows rows of x (both blocks
// of a pair together) and 2 BN rows of weights per K step, and the launch
// takes ceil(tiles / slots) rounds of such tiles.  Pick the width whose rounds
// move the fewest rows (the widest on a tie).  Measured on GB300: with 152 SMs
// and I = 14336, M <= 128 gets 96 (150 tiles in one round, fewer weight rows
// per block than 128); M = 8192 gets 128 where a rule on columns alone picked
// 64 for 1 % less wave quantisation and ran 1.8 times slower.
int pick_bn(int64_t m_blocks, int64_t I, int64_t slots, int64_t a_rows, int cols_per_bn = 1)
{
    if (I <= 64 * cols_per_bn) return 64;
    int best = 128;
    int64_t best_cost = -1;
    for (int bn : {128, 96, 64}) {
        const int64_t tiles = m_blocks * ((I + cols_per_bn * bn - 1) / (cols_per_bn * bn));
        const int64_t cost = (tiles + slots - 1) / slots * (a_rows + 2 * bn);
        if (best_cost < 0 || cost < best_cost) {
            best = bn;
            best_cost = cost;
        }
    }
    return best;
}

// Per kernel variant and device: the shared-memory opt-in done, and how many
// blocks (one shape) or pairs (the other) fit on the GPU at once.
constexpr int kMaxDevices = 64;
std::atomic<int> g_slots[kMaxDevices][2][5][6];     // [device][bf16][activation, 4 = plain][variant]

bool overlap(uintptr_t a0, uint64_t alen, uintptr_t b0, uint64_t blen)
{
    return a0 < b0 + blen && b0 < a0 + alen;
}

}  // namespace

cudaError_t timeouts(unsigned int *count, bool reset)
{
    cudaError_t e = cudaMemcpyFromSymbol(count, g_gemm_timeouts, sizeof(unsigned int));
    if (e == cudaSuccess && reset) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_gemm_timeouts, &zero, sizeof(unsigned int));
    }
    return e;
}

}  // namespace gemm
}  // namespace glu

namespace glu {
namespace gemm {
namespace {

// glu_gemm_fwd (act 0..3: y = act(x w_gate^T) * (x w_up^T), I output columns)
// and glu_gemm_nt (act 4: y = x w^T with w_gate = w_up = w, I = its rows).
int run_gemm(const void *x, int64_t x_stride, const void *w_gate, const void *w_up, int64_t w_stride, void *y,
             int64_t y_stride, int64_t M, int64_t K, int64_t I, int act, glu_dtype_t dtype, glu_stream_t stream)
{
    const bool plain = act == kPlainAct;
    if (act < GLU_ACT_SILU || act > kPlainAct || (dtype != GLU_F16 && dtype != GLU_BF16)) return GLU_ERR_ENUM;
    if (M < 0 || K < 0 || I < 0 || M > INT32_MAX || K > INT32_MAX || I > INT32_MAX) return GLU_ERR_SHAPE;
    if (M == 0 || I == 0) {
        glu::record_launch(glu_launch_info_t{});
        return GLU_OK;
    }
    if (!y || (K > 0 && (!x || !w_gate || !w_up))) return GLU_ERR_NULL;
    const int E = 2;
    if (y_stride < I || (K > 0 && (x_stride < K || w_stride < K))) return GLU_ERR_STRIDE;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint64_t ylen = (uint64_t(M - 1) * uint64_t(y_stride) + uint64_t(I)) * E;
    if (K == 0) {   // empty sums: y = act(0) * 0 = 0
        cudaError_t e = cudaMemset2DAsync(y, size_t(y_stride) * E, 0, size_t(I) * E, size_t(M), s);
        if (e != cudaSuccess) return glu::cuda_fail(e);
        glu::record_launch(glu_launch_info_t{});
        return GLU_OK;
    }
    // the tensor-memory accelerator needs 16-byte aligned bases and row strides
    if (uintptr_t(x) % 16 || uintptr_t(w_gate) % 16 || uintptr_t(w_up) % 16 || (x_stride * E) % 16 ||
        (w_stride * E) % 16)
        return GLU_ERR_STRIDE;
    const uint64_t xlen = (uint64_t(M - 1) * uint64_t(x_stride) + uint64_t(K)) * E;
    const uint64_t wlen = (uint64_t(I - 1) * uint64_t(w_stride) + uint64_t(K)) * E;
    if (overlap(uintptr_t(y), ylen, uintptr_t(x), xlen) || overlap(uintptr_t(y), ylen, uintptr_t(w_gate), wlen) ||
        overlap(uintptr_t(y), ylen, uintptr_t(w_up), wlen))
        return GLU_ERR_ALIAS;

    // the tensor-memory accelerator is given device memory only: an operand
    // anywhere else (pinned host memory included) is refused before launch
    for (const void *q : {x, w_gate, w_up, static_cast<const void *>(y)}) {
        bool dev_mem = false;
        const cudaError_t pe = glu::on_device(q, &dev_mem);
        if (pe != cudaSuccess) return glu::cuda_fail(pe);
        if (!dev_mem) return GLU_ERR_VALUE;
    }
    const bool bf16 = dtype == GLU_BF16;
    const int ctas = M > BM ? 2 : 1;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) { (void)cudaGetLastError(); return glu::cuda_fail(e); }
    const int64_t rows_per_block = int64_t(BM) * ctas;
    const int64_t tile_rows = ctas == 1 ? (M + 7) / 8 * 8 : rows_per_block;     // rows of x a tile loads
    const int bn = pick_bn((M + rows_per_block - 1) / rows_per_block, I, sms / ctas, tile_rows, plain ? 2 : 1);
    const Variant v = pick(bf16, act, bn, ctas);

    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = unsigned(ctas);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = size_t(v.smem);
    cfg.stream = s;

    std::atomic<int> &slots = g_slots[dev % kMaxDevices][bf16][act][v.id];
    int n_slots = slots.load(std::memory_order_acquire);
    if (n_slots == 0) {
        e = cudaFuncSetAttribute(reinterpret_cast<const void *>(v.fn), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 v.smem);
        if (e != cudaSuccess) { (void)cudaGetLastError(); return glu::cuda_fail(e); }
        n_slots = sms;
        if (ctas > 1) {
            cudaLaunchConfig_t q = cfg;
            q.gridDim = dim3(unsigned(sms - sms % ctas));
            q.attrs = &attr[1];
            q.numAttrs = 1;
            int clusters = 0;
            e = cudaOccupancyMaxActiveClusters(&clusters, reinterpret_cast<const void *>(v.fn), &q);
            if (e != cudaSuccess || clusters <= 0) {
                (void)cudaGetLastError();
                clusters = sms / ctas;
            }
            n_slots = clusters;
        }
        slots.store(n_slots, std::memory_order_release);
    }

    const bool y_aligned = (uintptr_t(y) % 16 == 0) && ((y_stride * E) % 16 == 0);
    CUtensorMap tx, tg, tu, ty;
    // one block holding every row copies only the rows that exist (rounded up to
    // a swizzle atom of 8): the MMA rows past them read stale shared memory and
    // produce accumulator rows that are never stored
    const int a_rows = ctas == 1 ? int((M + 7) / 8 * 8) : BM;
    if (!make_map(&tx, bf16, x, M, K, x_stride * E, BK, a_rows, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&tg, bf16, w_gate, I, K, w_stride * E, BK, bn, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&tu, bf16, w_up, I, K, w_stride * E, BK, bn, CU_TENSOR_MAP_SWIZZLE_128B))
        return glu::cuda_fail(cudaErrorInvalidValue);
    // y through the copy engine when its rows allow, else direct stores (the map is then
    // unused).  The engine clips a box at y's last column in 16-byte units, so the
    // row width must be a whole number of them.
    const bool y_map = y_aligned && (I * E) % 16 == 0 &&
                       make_map(&ty, bf16, y, M, I, y_stride * E, kYBox, kYBox, CU_TENSOR_MAP_SWIZZLE_64B);
    if (!y_map) ty = tx;

    Params p{};
    p.y = static_cast<char *>(y);
    p.y_stride = y_stride * E;
    p.M = int(M);
    p.I = int(I);
    p.K = int(K);
    p.k_tiles = int((K + BK - 1) / BK);
    p.m_blocks = int((M + rows_per_block - 1) / rows_per_block);
    p.i_blocks = int((I + (plain ? 2 : 1) * bn - 1) / ((plain ? 2 : 1) * bn));
    // row blocks per group: their x rows (about 48 MiB at most) stay in L2
    // while the weight slices stream past them once
    const int64_t block_bytes = rows_per_block * K * E;
    int64_t group = (int64_t(48) << 20) / block_bytes;
    group = group < 1 ? 1 : (group > p.m_blocks ? p.m_blocks : group);
    p.group_m = int(group);
    p.vec_store = y_aligned;
    p.a_bytes = uint32_t(a_rows) * BK * E;
    p.tma_store = y_map;
    const int64_t tiles = int64_t(p.m_blocks) * p.i_blocks;
    if (tiles * ctas > INT32_MAX) return GLU_ERR_SHAPE;
    const int64_t clusters = tiles < n_slots ? tiles : n_slots;     // persistent

    void *args[] = {&tx, &tg, &tu, &ty, &p};
    cfg.gridDim = dim3(unsigned(clusters * ctas));
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(v.fn), args);
    if (e != cudaSuccess) {     // retry without the dependent-launch attribute
        (void)cudaGetLastError();
        cfg.attrs = &attr[1];
        cfg.numAttrs = 1;
        e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(v.fn), args);
    }
    if (e != cudaSuccess) { (void)cudaGetLastError(); return glu::cuda_fail(e); }
    glu_launch_info_t info{};
    info.launched = 1;
    info.vec_bytes = p.tma_store ? 2 * kYBox : (p.vec_store ? 16 : E);
    info.unroll = ctas;
    info.threads = kThreads;
    info.grid = int32_t(clusters * ctas);
    info.path = plain ? 5 : 3;
    info.vector_units = tiles;
    glu::record_launch(info);
    return GLU_OK;
}

}  // namespace
}  // namespace gemm
}  // namespace glu

extern "C" int glu_gemm_fwd(const void *x, int64_t x_stride, const void *w_gate, const void *w_up,
                            int64_t w_stride, void *y, int64_t y_stride, int64_t M, int64_t K, int64_t I,
                            glu_act_t act, glu_dtype_t dtype, glu_stream_t stream)
{
    if (act < GLU_ACT_SILU || act > GLU_ACT_RELU) return GLU_ERR_ENUM;
    return glu::gemm::run_gemm(x, x_stride, w_gate, w_up, w_stride, y, y_stride, M, K, I, act, dtype, stream);
}

extern "C" int glu_gemm_nt(const void *a, int64_t a_stride, const void *b, int64_t b_stride, void *d,
                           int64_t d_stride, int64_t M, int64_t K, int64_t N, glu_dtype_t dtype, glu_stream_t stream)
{
    return glu::gemm::run_gemm(a, a_stride, b, b, b_stride, d, d_stride, M, K, N, glu::gemm::kPlainAct, dtype,
                               stream);
}

// ---------------------------------------------------------------- the gated MLP

namespace glu {
namespace gemm {
namespace {

// The rows run in chunks of at most this many bytes of y.  Measured on GB300
// (4096 x 4096 x 14336, bf16): chunks of 1536 rows, whose 44 MiB of y stay in
// L2 between the two products, took 0.847 ms; the whole batch in one chunk,
// y through HBM, 0.778 ms: launches of fewer rows lose more to tile rounds and
// pipeline fill than the 2 x 117 MB of y traffic cost.  So a chunk is as large
// as the workspace allows, and the default workspace holds the whole y up to
// this cap.
constexpr uint64_t kMlpChunkBytes = uint64_t(1) << 30;

int64_t round_up8(int64_t v) { return (v + 7) / 8 * 8; }

// Rows of y a chunk holds within `bytes`: whole 256-row blocks of the pair
// shape when more than 256 rows fit, else as many rows as fit; at most M.
int64_t mlp_chunk_rows(int64_t M, int64_t I, uint64_t bytes)
{
    const uint64_t row = uint64_t(round_up8(I)) * 2;
    int64_t rows = int64_t(bytes / row);
    if (rows > 256) rows = rows / 256 * 256;
    return rows < M ? rows : M;
}

}  // namespace
}  // namespace gemm
}  // namespace glu

extern "C" size_t glu_mlp_workspace_bytes(int64_t M, int64_t I, glu_dtype_t dtype)
{
    using namespace glu::gemm;
    if (M <= 0 || I <= 0 || I > INT32_MAX || (dtype != GLU_F16 && dtype != GLU_BF16)) return 0;
    return size_t(mlp_chunk_rows(M, I, kMlpChunkBytes)) * size_t(round_up8(I)) * 2;
}

extern "C" int glu_mlp_fwd(const void *x, int64_t x_stride, const void *w_gate, const void *w_up, int64_t w_stride,
                           const void *w_down, int64_t w_down_stride, void *out, int64_t out_stride, int64_t M,
                           int64_t H, int64_t I, glu_act_t act, glu_dtype_t dtype, void *workspace,
                           size_t workspace_bytes, glu_stream_t stream)
{
    using namespace glu::gemm;
    if (act < GLU_ACT_SILU || act > GLU_ACT_RELU || (dtype != GLU_F16 && dtype != GLU_BF16)) return GLU_ERR_ENUM;
    if (M < 0 || H < 0 || I < 0 || M > INT32_MAX || H > INT32_MAX || I > INT32_MAX) return GLU_ERR_SHAPE;
    if (M == 0 || H == 0) {
        glu::record_launch(glu_launch_info_t{});
        return GLU_OK;
    }
    if (!out || !x || !w_gate || !w_up || (I > 0 && !w_down)) return GLU_ERR_NULL;
    if (x_stride < H || w_stride < H || out_stride < H || (I > 0 && w_down_stride < I)) return GLU_ERR_STRIDE;
    const int E = 2;
    const int64_t ys = round_up8(I);            // the chunk's y rows, 16-byte multiples for the copy engine
    if (I > 0) {
        if (!workspace || workspace_bytes < uint64_t(ys) * E) return GLU_ERR_WORKSPACE;
        // every operand goes through the tensor-memory accelerator: 16-byte
        // aligned bases and row strides, device memory, checked before the
        // first launch
        if (uintptr_t(workspace) % 16 || uintptr_t(x) % 16 || uintptr_t(w_gate) % 16 || uintptr_t(w_up) % 16 ||
            uintptr_t(w_down) % 16 || (x_stride * E) % 16 || (w_stride * E) % 16 || (w_down_stride * E) % 16)
            return GLU_ERR_STRIDE;
    }
    // out is written while x is still being read (by later chunks): no overlap
    // with any operand or the workspace
    const uint64_t olen = (uint64_t(M - 1) * uint64_t(out_stride) + uint64_t(H)) * E;
    const uint64_t xlen = (uint64_t(M - 1) * uint64_t(x_stride) + uint64_t(H)) * E;
    const uint64_t wlen = I > 0 ? (uint64_t(I - 1) * uint64_t(w_stride) + uint64_t(H)) * E : 0;
    const uint64_t dlen = I > 0 ? (uint64_t(H - 1) * uint64_t(w_down_stride) + uint64_t(I)) * E : 0;
    if (overlap(uintptr_t(out), olen, uintptr_t(x), xlen) || overlap(uintptr_t(out), olen, uintptr_t(w_gate), wlen) ||
        overlap(uintptr_t(out), olen, uintptr_t(w_up), wlen) || overlap(uintptr_t(out), olen, uintptr_t(w_down), dlen) ||
        (I > 0 && overlap(uintptr_t(out), olen, uintptr_t(workspace), workspace_bytes)))
        return GLU_ERR_ALIAS;
    if (I > 0) {
        for (const void *q : {x, w_gate, w_up, w_down, static_cast<const void *>(workspace),
                              static_cast<const void *>(out)}) {
            bool dev_mem = false;
            const cudaError_t pe = glu::on_device(q, &dev_mem);
            if (pe != cudaSuccess) return glu::cuda_fail(pe);
            if (!dev_mem) return GLU_ERR_VALUE;
        }
    }
    if (I == 0) {           // empty inner sums: out = 0
        cudaError_t e = cudaMemset2DAsync(out, size_t(out_stride) * E, 0, size_t(H) * E, size_t(M),
                                          reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return glu::cuda_fail(e);
        glu::record_launch(glu_launch_info_t{});
        return GLU_OK;
    }
    const uint64_t budget = workspace_bytes < kMlpChunkBytes ? workspace_bytes : kMlpChunkBytes;
    const int64_t chunk = mlp_chunk_rows(M, I, budget);
    for (int64_t r0 = 0; r0 < M; r0 += chunk) {
        const int64_t rows = M - r0 < chunk ? M - r0 : chunk;
        const char *xr = static_cast<const char *>(x) + r0 * x_stride * E;
        char *outr = static_cast<char *>(out) + r0 * out_stride * E;
        int st = glu_gemm_fwd(xr, x_stride, w_gate, w_up, w_stride, workspace, ys, rows, H, I, act, dtype, stream);
        if (st != GLU_OK) return st;
        st = glu_gemm_nt(workspace, ys, w_down, w_down_stride, outr, out_stride, rows, I, H, dtype, stream);
        if (st != GLU_OK) return st;
    }
    return GLU_OK;
}
