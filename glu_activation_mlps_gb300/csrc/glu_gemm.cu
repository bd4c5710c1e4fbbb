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
// A persistent grid of one block per SM walks 128 x BN tiles of y.  Warp 0
// moves 64-wide K slices of x, w_gate and w_up into a ring of shared-memory
// stages with the tensor-memory accelerator (128-byte swizzle); the gate and
// up slices sit back to back, so one tcgen05.mma of N = 2 BN (kind::f16,
// M = 128, K = 16), issued by one thread of warp 1, accumulates both into one
// fp32 [gate | up] block of tensor memory.  Tensor memory holds two such
// blocks, so the MMAs of the next tile run while warps 2-5 read the finished
// one with tcgen05.ld (one row per thread), apply the same fp32 activation as
// the streaming kernels, round once and store.  Tiles are ordered in groups of
// eight row blocks so that weight slices are reused from L2 by the blocks
// running at the same time.
//
// Every wait is bounded by a clock budget (about a second); a wait that runs
// out is counted in a device word (read by glu_wait_timeouts) and raises a
// block-wide abort flag: every role leaves its loop, the producer and the MMA
// issuer wait (bounded) for the copies and MMAs already issued, the block
// frees its tensor memory and returns with the remaining tiles unwritten.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "glu.h"
#include "glu_kernels.cuh"
#include "glu_plan.h"

namespace glu {
namespace gemm {

constexpr int BM = 128;                  // rows of x per tile (tensor-memory lanes)
constexpr int BK = 64;                   // K per stage: 64 x 2 bytes = one 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kThreads = 192;            // warp 0 loads, warp 1 issues MMAs, warps 2-5 store
constexpr int kEpiWarps = 4;
constexpr long long kBudget = 2000000000LL;   // ~1 s at 2 GHz
constexpr int kGroupM = 8;

template <int BN>
struct Shape {
    static constexpr int kTileA = BM * BK * 2;
    static constexpr int kTileB = BN * BK * 2;                    // one of gate, up
    static constexpr int kStageBytes = kTileA + 2 * kTileB;
    static constexpr int kAccCols = 2 * BN;                       // [gate | up] of one tile
    static constexpr int kTmemCols = 2 * kAccCols;                // two tiles in flight
    static constexpr int kBars = 2 * kStages + 2 + 2 + 1;         // full, empty, acc_full, acc_empty, done
    static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kBars * 8 + 16;
    static_assert(BN % 32 == 0 && BN >= 32 && 2 * BN <= 256, "one MMA covers N = 2 BN <= 256");
    static_assert(kTmemCols <= 512, "tensor memory holds 512 columns");
    static_assert(kTileA % 1024 == 0 && kTileB % 1024 == 0, "swizzle atoms stay 1024-byte aligned");
};

struct Params {
    char *y;
    int64_t y_stride;       // bytes
    int M, I, K;
    int k_tiles;
    int m_blocks, i_blocks;
    int vec_store;          // y rows and base 16-byte aligned
};

static __device__ unsigned int g_gemm_timeouts;

__device__ __forceinline__ uint32_t saddr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool wait_parity(uint32_t bar, uint32_t parity)
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
        if (clock64() - t0 > kBudget) return false;
    }
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

__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
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

__device__ __forceinline__ void arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Tile t of the grouped order: eight row blocks side by side walk the column blocks.
__device__ __forceinline__ void tile_origin(const Params &p, int t, int &m0, int &ib)
{
    const int per_group = kGroupM * p.i_blocks;
    const int first_m = (t / per_group) * kGroupM;
    const int gsize = min(p.m_blocks - first_m, kGroupM);
    const int r = t % per_group;
    m0 = (first_m + r % gsize) * BM;
    ib = r / gsize;
}

template <class Act, class T, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    glu_gemm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_wg,
                    const __grid_constant__ CUtensorMap tm_wu, const Params p)
{
    using S = Shape<BN>;
    using Cd = Codec<T>;
    constexpr uint32_t kIdesc = idesc_f16(std::is_same<T, __nv_bfloat16>::value ? 1 : 0, BM, 2 * BN);

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = saddr(smem_raw);
    unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);     // 1024-byte aligned ring
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * S::kStageBytes);
    uint64_t *empty = full + kStages;
    uint64_t *acc_full = empty + kStages;       // [2]: MMAs of a tile done
    uint64_t *acc_empty = acc_full + 2;         // [2]: the epilogue has read a tile
    uint64_t *done = acc_empty + 2;             // every MMA this block issued, done
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(done + 1) + 1;

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles = p.m_blocks * p.i_blocks;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&full[s])) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&empty[s])) : "memory");
        }
        for (int b = 0; b < 2; ++b) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&acc_full[b])) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(&acc_empty[b])), "r"(kEpiWarps)
                         : "memory");
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(done)) : "memory");
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         saddr(const_cast<uint32_t *>(tmem_slot))),
                     "r"(S::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == 0) {
        if (lane == 0) {
            // producer: stage s = it % kStages is reused for the (it / kStages)-th time
            uint32_t it = 0;
            for (int t = blockIdx.x; t < n_tiles && !*abort_flag; t += gridDim.x) {
                int m0, ib;
                tile_origin(p, t, m0, ib);
                const int i0 = ib * BN;
                for (int kt = 0; kt < p.k_tiles; ++kt, ++it) {
                    const uint32_t s = it % kStages, use = it / kStages;
                    if (*abort_flag) break;
                    if (use > 0 && !wait_parity(saddr(&empty[s]), (use - 1) & 1)) {
                        atomicAdd(&g_gemm_timeouts, 1u);
                        *abort_flag = 1;
                        break;
                    }
                    unsigned char *st = smem + s * S::kStageBytes;
                    const uint32_t bar = saddr(&full[s]);
                    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                                 "r"(uint32_t(S::kStageBytes))
                                 : "memory");
                    tma_load(saddr(st), &tm_x, kt * BK, m0, bar);
                    tma_load(saddr(st + S::kTileA), &tm_wg, kt * BK, i0, bar);
                    tma_load(saddr(st + S::kTileA + S::kTileB), &tm_wu, kt * BK, i0, bar);
                }
            }
            // the block may only exit once every copy it issued has landed
            const uint32_t first = it > uint32_t(kStages) ? it - kStages : 0;
            for (uint32_t j = first; j < it; ++j)
                if (!wait_parity(saddr(&full[j % kStages]), (j / kStages) & 1)) {
                    atomicAdd(&g_gemm_timeouts, 1u);
                    break;
                }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t it = 0;
            int lt = 0;
            for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++lt) {
                if (*abort_flag) break;
                const int ab = lt & 1, use_acc = lt >> 1;
                if (use_acc > 0 && !wait_parity(saddr(&acc_empty[ab]), (use_acc - 1) & 1)) {
                    atomicAdd(&g_gemm_timeouts, 1u);
                    *abort_flag = 1;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t d = tmem + uint32_t(ab * S::kAccCols);
                bool ok = true;
                for (int kt = 0; kt < p.k_tiles; ++kt, ++it) {
                    const uint32_t s = it % kStages, use = it / kStages;
                    if (!wait_parity(saddr(&full[s]), use & 1)) {
                        atomicAdd(&g_gemm_timeouts, 1u);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t a0 = saddr(smem + s * S::kStageBytes);
                    const uint64_t da = desc_sw128(a0);
                    const uint64_t db = desc_sw128(a0 + S::kTileA);    // gate rows, then up rows
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        // K advances by 16 elements = 32 bytes inside the swizzle row
                        const uint64_t step = uint64_t(kk * 32 >> 4);
                        mma(d, da + step, db + step, kIdesc, (kt | kk) != 0);
                    }
                    mma_commit(saddr(&empty[s]));       // the stage is free once these MMAs finish
                }
                if (!ok) break;
                mma_commit(saddr(&acc_full[ab]));       // the tile's accumulator is complete
            }
            mma_commit(saddr(done));
            if (!wait_parity(saddr(done), 0)) atomicAdd(&g_gemm_timeouts, 1u);
        }
    } else {
        // epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. +31, one row per thread
        const int q = warp & 3;
        const uint32_t lane_base = uint32_t(q * 32) << 16;
        int lt = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++lt) {
            if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) break;
            const int ab = lt & 1, use_acc = lt >> 1;
            // tcgen05.ld is warp-collective: the whole warp takes one decision
            const bool ok = __all_sync(0xFFFFFFFFu, wait_parity(saddr(&acc_full[ab]), use_acc & 1));
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            if (!ok) {
                if (lane == 0) {
                    atomicAdd(&g_gemm_timeouts, 1u);
                    *abort_flag = 1;
                }
                break;
            }
            int m0, ib;
            tile_origin(p, t, m0, ib);
            const int m = m0 + q * 32 + lane;
            const int i0 = ib * BN;
            const uint32_t acc = tmem + lane_base + uint32_t(ab * S::kAccCols);
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t g[32], u[32];
                tmem_ld32(acc + uint32_t(c0), g);
                tmem_ld32(acc + uint32_t(BN + c0), u);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                if (c0 + 32 == BN) {          // all of this tile read: hand the accumulator back
                    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) arrive(saddr(&acc_empty[ab]));
                }
                if (m >= p.M) continue;
                uint32_t packed[32 / Cd::kPerWord];
#pragma unroll
                for (int j = 0; j < 32; j += Cd::kPerWord) {
                    float f[Cd::kPerWord];
#pragma unroll
                    for (int e = 0; e < Cd::kPerWord; ++e)
                        f[e] = op_fwd<Act, false>(__uint_as_float(g[j + e]), __uint_as_float(u[j + e]));
                    packed[j / Cd::kPerWord] = Cd::put(f);
                }
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
                            Cd::store1(dst + j * int64_t(sizeof(T)), Cd::get(packed[j / Cd::kPerWord], j % Cd::kPerWord));
                    }
                }
            }
        }
    }

    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(S::kTmemCols)
                     : "memory");
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
// whose box is 64 columns by `box_rows` rows, 128-byte swizzle, zero fill
// outside the matrix.
bool make_map(CUtensorMap *m, bool bf16, const void *base, int64_t rows, int64_t cols, int64_t stride_bytes,
              int box_rows)
{
    EncodeFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(stride_bytes)};
    const cuuint32_t box[2] = {cuuint32_t(BK), cuuint32_t(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

using KernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, Params);

template <class T, int BN>
KernelFn pick(int act)
{
    switch (act) {
    case 0: return glu_gemm_kernel<Silu, T, BN>;
    case 1: return glu_gemm_kernel<GeluErf, T, BN>;
    case 2: return glu_gemm_kernel<GeluTanh, T, BN>;
    case 3: return glu_gemm_kernel<Relu, T, BN>;
    default: return nullptr;
    }
}

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

extern "C" int glu_gemm_fwd(const void *x, int64_t x_stride, const void *w_gate, const void *w_up,
                            int64_t w_stride, void *y, int64_t y_stride, int64_t M, int64_t K, int64_t I,
                            glu_act_t act, glu_dtype_t dtype, glu_stream_t stream)
{
    using namespace glu::gemm;
    if (act < GLU_ACT_SILU || act > GLU_ACT_RELU || (dtype != GLU_F16 && dtype != GLU_BF16)) return GLU_ERR_ENUM;
    if (M < 0 || K < 0 || I < 0 || M > INT32_MAX || K > INT32_MAX || I > INT32_MAX) return GLU_ERR_SHAPE;
    if (M == 0 || I == 0) return GLU_OK;
    if (!y || (K > 0 && (!x || !w_gate || !w_up))) return GLU_ERR_NULL;
    const int E = 2;
    if (y_stride < I || (K > 0 && (x_stride < K || w_stride < K))) return GLU_ERR_STRIDE;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint64_t ylen = (uint64_t(M - 1) * uint64_t(y_stride) + uint64_t(I)) * E;
    if (K == 0) {   // empty sums: y = act(0) * 0 = 0
        cudaError_t e = cudaMemset2DAsync(y, size_t(y_stride) * E, 0, size_t(I) * E, size_t(M), s);
        return e == cudaSuccess ? GLU_OK : glu::cuda_fail(e);
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

    const bool bf16 = dtype == GLU_BF16;
    const int bn = I <= 64 ? 64 : 128;
    KernelFn fn = bn == 64 ? (bf16 ? pick<__nv_bfloat16, 64>(act) : pick<__half, 64>(act))
                           : (bf16 ? pick<__nv_bfloat16, 128>(act) : pick<__half, 128>(act));
    const int smem = bn == 64 ? Shape<64>::kSmemBytes : Shape<128>::kSmemBytes;
    static std::atomic<int> smem_set[2][4][2];
    std::atomic<int> &flag = smem_set[bf16][act][bn == 128];
    if (!flag.load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void *>(fn),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) { (void)cudaGetLastError(); return glu::cuda_fail(e); }
        flag.store(1, std::memory_order_release);
    }

    CUtensorMap tx, tg, tu;
    if (!make_map(&tx, bf16, x, M, K, x_stride * E, BM) || !make_map(&tg, bf16, w_gate, I, K, w_stride * E, bn) ||
        !make_map(&tu, bf16, w_up, I, K, w_stride * E, bn))
        return glu::cuda_fail(cudaErrorInvalidValue);

    Params p{};
    p.y = static_cast<char *>(y);
    p.y_stride = y_stride * E;
    p.M = int(M);
    p.I = int(I);
    p.K = int(K);
    p.k_tiles = int((K + BK - 1) / BK);
    p.m_blocks = int((M + BM - 1) / BM);
    p.i_blocks = int((I + bn - 1) / bn);
    p.vec_store = (uintptr_t(y) % 16 == 0) && ((y_stride * E) % 16 == 0);
    const int64_t tiles = int64_t(p.m_blocks) * p.i_blocks;
    if (tiles > INT32_MAX) return GLU_ERR_SHAPE;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) { (void)cudaGetLastError(); return glu::cuda_fail(e); }
    const int64_t blocks = tiles < sms ? tiles : sms;     // persistent: one block per SM

    void *args[] = {&tx, &tg, &tu, &p};
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = size_t(smem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(fn), args);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        cfg.attrs = nullptr;
        cfg.numAttrs = 0;
        e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(fn), args);
    }
    if (e != cudaSuccess) { (void)cudaGetLastError(); return glu::cuda_fail(e); }
    return GLU_OK;
}
