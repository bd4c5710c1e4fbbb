// Fused residual add + RMSNorm ("Skill: Write a Triton Fused Add+RMSNorm
// Kernel": Purpose; Required reasoning process steps 1-9; Kernel design rules;
// Correctness requirements):
//
//     s = x + residual (fp32),  h = round(s),
//     rstd = 1 / sqrt(sum(s^2) / H + eps),  y = round(s * rstd * gamma)
//
// One block per row (more rows than blocks: the grid walks them).  Each thread
// keeps EPT elements of s in fp32 registers, so x and the residual are read
// once and h and y written once: 4 row passes of HBM traffic plus gamma, which
// stays in L2 ("Performance requirements": the single-pass case).  Every
// element is loaded and stored by one thread, its loads before its stores, and
// y is stored only after the whole block has loaded its row, which makes h or
// y written over x or the residual safe.  The sum of squares is formed with
// fused multiply-adds in partial sums of 8 elements per thread, then reduced
// over the warp and the block in fp32; rstd uses IEEE division and square root.
//
// Rows whose operands are 16-byte aligned (bases, strides and row width) use
// 16-byte accesses, element i of a thread's k-th vector at column
// (t + k * threads) * V + i: rows of 16 KiB or more in a persistent grid
// (add_rmsnorm_rows_kernel), narrower ones one block per row
// (add_rmsnorm_kernel); other rows use element accesses at column
// t + k * threads, one block per row.  Either way consecutive threads touch
// consecutive addresses.
//
// The backward (glu_add_rmsnorm_bwd, below the forward) has four kernels, for
// 16-byte rows in device memory: add_rmsnorm_bwd_narrow_kernel for narrow rows
// when its grid fits on the GPU at once, add_rmsnorm_bwd_teams_kernel (a
// persistent grid of register teams) for other rows of up to 512 vectors
// (384 for f32), and
// add_rmsnorm_bwd_staged_kernel (rows staged in shared memory by the
// bulk-copy engine) for wider ones; add_rmsnorm_bwd_kernel with element
// accesses takes the rest.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "glu.h"
#include "glu_async.cuh"
#include "glu_kernels.cuh"
#include "glu_internal.h"

namespace glu {
namespace rms {

struct Params {
    const char *x, *res, *gamma;
    char *h, *y;
    float *rstd;
    int64_t sx, sr, sh, sy;     // row strides in bytes
    int64_t rows;
    int H;
    float eps;
    int prefetch;               // 16-byte rows: ask L2 for the block's first row before the dependency wait
};

// An L2 prefetch of `bytes` bytes at q by the bulk-copy engine (q 16-byte
// aligned, bytes a multiple of 16).  Used before a kernel waits for the
// previous grid: L2 is the point of coherence, so a line that grid writes
// after the prefetch is simply fetched again, and nothing enters the core's
// own caches before the wait.
__device__ __forceinline__ void prefetch_bulk(const void *q, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(q), "r"(bytes) : "memory");
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Sum of v over the block; every thread gets the result.  `red` holds 33
// floats; consecutive rows alternate between two such arrays, so the array a
// row reads is not written again until every thread has passed the next row's
// first barrier.
__device__ __forceinline__ float block_sum(float v, float *red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_sum(v);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float w = lane < nw ? red[lane] : 0.0f;
        w = warp_sum(w);
        if (lane == 0) red[32] = w;
    }
    __syncthreads();
    return red[32];
}

// Sum of squares of a thread's elements: fused multiply-adds into partial sums
// of (at most) 8 elements each, added pairwise at the end.  With the 5 + 5
// additions of the warp and block reduction, every sum a block forms carries at
// most 8 + 3 + 10 = 21 fp32 roundings of non-negative terms.
template <int N>
struct SumSq {
    static constexpr int P = N / 8 > 0 ? N / 8 : 1;
    float part[P];
    __device__ __forceinline__ SumSq()
    {
#pragma unroll
        for (int i = 0; i < P; ++i) part[i] = 0.0f;
    }
    __device__ __forceinline__ void add(int i, float f) { part[(i / 8) % P] = fmaf(f, f, part[(i / 8) % P]); }
    __device__ __forceinline__ void add(int i, float a, float b) { part[(i / 8) % P] = fmaf(a, b, part[(i / 8) % P]); }
    __device__ __forceinline__ float total() const
    {
        float q[P];
#pragma unroll
        for (int i = 0; i < P; ++i) q[i] = part[i];
#pragma unroll
        for (int w = 1; w < P; w *= 2)
#pragma unroll
            for (int i = 0; i + w < P; i += 2 * w) q[i] += q[i + w];
        return q[0];
    }
};

template <class T, int EPT, bool VEC>
__global__ void __launch_bounds__(EPT <= 16 ? 1024 : 512)
    add_rmsnorm_kernel(const Params p)
{
    using C = Codec<T>;
    constexpr int V = VEC ? 16 / int(sizeof(T)) : 1;      // elements per access
    constexpr int NV = EPT / V;                           // accesses per thread per operand
    constexpr int W = V / C::kPerWord > 0 ? V / C::kPerWord : 1;   // 32-bit words per access
    __shared__ float red[2][33];

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // the block's first row of x and the residual, asked of L2 before the wait
    if (VEC && p.prefetch && threadIdx.x == 0 && blockIdx.x < p.rows) {
        prefetch_bulk(p.x + int64_t(blockIdx.x) * p.sx, uint32_t(p.H) * sizeof(T));
        prefetch_bulk(p.res + int64_t(blockIdx.x) * p.sr, uint32_t(p.H) * sizeof(T));
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const int t = threadIdx.x, nt = blockDim.x;
    int parity = 0;
    for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x, parity ^= 1) {
        const char *xr = p.x + row * p.sx, *rr = p.res + row * p.sr;
        char *hr = p.h + row * p.sh, *yr = p.y + row * p.sy;
        float s[EPT];
        SumSq<EPT> ss;
        // loads go out in chunks of CK accesses per operand, all of a chunk's
        // loads before its stores (each element is loaded and stored by this
        // thread alone, so h over x or the residual stays correct)
        if constexpr (VEC) {
            constexpr int CK = NV < 4 ? NV : 4;
#pragma unroll
            for (int k0 = 0; k0 < NV; k0 += CK) {
                uint32_t wx[CK][W], wr[CK][W];
#pragma unroll
                for (int k = 0; k < CK; ++k) {
                    const int col = (t + (k0 + k) * nt) * V;
                    if (col < p.H) {
                        Access<16>::load(xr + int64_t(col) * sizeof(T), reinterpret_cast<uint32_t(&)[4]>(wx[k]));
                        Access<16>::load(rr + int64_t(col) * sizeof(T), reinterpret_cast<uint32_t(&)[4]>(wr[k]));
                    }
                }
#pragma unroll
                for (int k = 0; k < CK; ++k) {
                    const int col = (t + (k0 + k) * nt) * V;
                    float *sv = s + (k0 + k) * V;
                    if (col < p.H) {
                        uint32_t wh[W];
#pragma unroll
                        for (int j = 0; j < W; ++j) {
                            float f[C::kPerWord];
#pragma unroll
                            for (int e = 0; e < C::kPerWord; ++e) {
                                f[e] = C::get(wx[k][j], e) + C::get(wr[k][j], e);
                                sv[j * C::kPerWord + e] = f[e];
                                ss.add((k0 + k) * V + j * C::kPerWord + e, f[e]);
                            }
                            wh[j] = C::put(f);
                        }
                        Access<16>::store(hr + int64_t(col) * sizeof(T), reinterpret_cast<const uint32_t(&)[4]>(wh));
                    } else {
#pragma unroll
                        for (int i = 0; i < V; ++i) sv[i] = 0.0f;
                    }
                }
            }
        } else {
            constexpr int CK = EPT < 8 ? EPT : 8;
#pragma unroll
            for (int k0 = 0; k0 < EPT; k0 += CK) {
                float xv[CK], rv[CK];
#pragma unroll
                for (int k = 0; k < CK; ++k) {
                    const int col = t + (k0 + k) * nt;
                    if (col < p.H) {
                        xv[k] = C::load1(xr + int64_t(col) * sizeof(T));
                        rv[k] = C::load1(rr + int64_t(col) * sizeof(T));
                    }
                }
#pragma unroll
                for (int k = 0; k < CK; ++k) {
                    const int col = t + (k0 + k) * nt;
                    s[k0 + k] = 0.0f;
                    if (col < p.H) {
                        s[k0 + k] = xv[k] + rv[k];
                        ss.add(k0 + k, s[k0 + k]);
                        C::store1(hr + int64_t(col) * sizeof(T), s[k0 + k]);
                    }
                }
            }
        }
        const float total = block_sum(ss.total(), red[parity]);
        const float rstd = 1.0f / sqrtf(total / float(p.H) + p.eps);
        if (t == 0 && p.rstd) p.rstd[row] = rstd;
        if constexpr (VEC) {
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int col = (t + k * nt) * V;
                if (col < p.H) {
                    uint32_t wg[W], wy[W];
                    Access<16>::load(p.gamma + int64_t(col) * sizeof(T), reinterpret_cast<uint32_t(&)[4]>(wg));
#pragma unroll
                    for (int j = 0; j < W; ++j) {
                        float f[C::kPerWord];
#pragma unroll
                        for (int e = 0; e < C::kPerWord; ++e)
                            f[e] = s[k * V + j * C::kPerWord + e] * rstd * C::get(wg[j], e);
                        wy[j] = C::put(f);
                    }
                    Access<16>::store(yr + int64_t(col) * sizeof(T), reinterpret_cast<const uint32_t(&)[4]>(wy));
                }
            }
        } else {
#pragma unroll
            for (int k = 0; k < EPT; ++k) {
                const int col = t + k * nt;
                if (col < p.H)
                    C::store1(yr + int64_t(col) * sizeof(T), s[k] * rstd * C::load1(p.gamma + int64_t(col) * sizeof(T)));
            }
        }
    }
}

// The 16-byte path as a persistent grid: every thread owns the same columns in
// every row, so gamma is read into registers once; the next row's x and
// residual are requested before this row's reduction starts, so a block always
// has loads in flight; s = x + residual is recomputed from the raw words for y
// (exact for 16-bit inputs, the same fp32 rounding for f32) instead of being
// held in registers.
template <class T, int EPT>
__global__ void __launch_bounds__(EPT <= 16 ? 1024 : 512)
    add_rmsnorm_rows_kernel(const Params p)
{
    using C = Codec<T>;
    constexpr int V = 16 / int(sizeof(T));
    constexpr int NV = EPT / V;
    constexpr int W = 4;
    __shared__ float red[2][33];

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // the block's first row of x and the residual, asked of L2 before the wait
    if (p.prefetch && threadIdx.x == 0 && blockIdx.x < p.rows) {
        prefetch_bulk(p.x + int64_t(blockIdx.x) * p.sx, uint32_t(p.H) * sizeof(T));
        prefetch_bulk(p.res + int64_t(blockIdx.x) * p.sr, uint32_t(p.H) * sizeof(T));
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const int t = threadIdx.x, nt = blockDim.x;
    bool on[NV];
    uint32_t gw[NV][W];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int col = (t + k * nt) * V;
        on[k] = col < p.H;
        if (on[k]) Access<16>::load(p.gamma + int64_t(col) * sizeof(T), gw[k]);
    }
    const auto load_row = [&](int64_t row, uint32_t (&wx)[NV][W], uint32_t (&wr)[NV][W]) {
        const char *xr = p.x + row * p.sx, *rr = p.res + row * p.sr;
#pragma unroll
        for (int k = 0; k < NV; ++k)
            if (on[k]) {
                const int64_t off = int64_t((t + k * nt) * V) * sizeof(T);
                Access<16>::load(xr + off, wx[k]);
                Access<16>::load(rr + off, wr[k]);
            }
    };

    uint32_t ax[NV][W], ar[NV][W];
    int64_t row = blockIdx.x;
    int parity = 0;
    if (row < p.rows) load_row(row, ax, ar);
    while (row < p.rows) {
        const int64_t next = row + gridDim.x;
        uint32_t bx[NV][W], br[NV][W];
        if (next < p.rows) load_row(next, bx, br);
        char *hr = p.h + row * p.sh, *yr = p.y + row * p.sy;
        SumSq<EPT> ss;
#pragma unroll
        for (int k = 0; k < NV; ++k)
            if (on[k]) {
                uint32_t wh[W];
#pragma unroll
                for (int j = 0; j < W; ++j) {
                    float f[C::kPerWord];
#pragma unroll
                    for (int e = 0; e < C::kPerWord; ++e) {
                        f[e] = C::get(ax[k][j], e) + C::get(ar[k][j], e);
                        ss.add(k * V + j * C::kPerWord + e, f[e]);
                    }
                    wh[j] = C::put(f);
                }
                Access<16>::store(hr + int64_t((t + k * nt) * V) * sizeof(T), wh);
            }
        const float total = block_sum(ss.total(), red[parity]);
        parity ^= 1;
        const float rstd = 1.0f / sqrtf(total / float(p.H) + p.eps);
        if (t == 0 && p.rstd) p.rstd[row] = rstd;
#pragma unroll
        for (int k = 0; k < NV; ++k)
            if (on[k]) {
                uint32_t wy[W];
#pragma unroll
                for (int j = 0; j < W; ++j) {
                    float f[C::kPerWord];
#pragma unroll
                    for (int e = 0; e < C::kPerWord; ++e)
                        f[e] = (C::get(ax[k][j], e) + C::get(ar[k][j], e)) * rstd * C::get(gw[k][j], e);
                    wy[j] = C::put(f);
                }
                Access<16>::store(yr + int64_t((t + k * nt) * V) * sizeof(T), wy);
            }
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int j = 0; j < W; ++j) {
                ax[k][j] = bx[k][j];
                ar[k][j] = br[k][j];
            }
        row = next;
    }
}

// ---------------------------------------------------------------- backward

struct BwdParams {
    const char *dy, *h, *gamma, *dh;
    const float *rstd;
    char *dx, *dres;
    float *dgamma;
    int64_t sdy, sh, sdh, sdx, sdr;     // row strides in bytes
    int64_t rows;
    int H;
    int tpr;                            // threads per row (a multiple of 32)
    int groups;                         // rows a block works on at once (staged kernel: teams)
    int stages;                         // staged kernel: shared-memory ring depth, in stages
};

// Waits of the staged backward that ran out, summed since the last reset.
static __device__ unsigned int g_rms_timeouts;

__device__ __forceinline__ void red_add_v4(float *p, float a, float b, float c, float d)
{
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

// The sum of v over the tpr threads of one row group; every thread of the
// group gets it.  `r` holds 33 floats, alternating between two arrays on
// consecutive rows like block_sum.  Warp sums, one barrier, then each thread
// adds its group's warp sums in order; for groups of more than 8 warps the
// group's first warp adds them and a second barrier shares the result.
__device__ __forceinline__ float group_sum(float v, float *r, int lane, int wig, int nwg)
{
    v = warp_sum(v);
    if (lane == 0) r[wig] = v;
    __syncthreads();
    if (nwg <= 8) {
        float t = 0.0f;
        for (int w = 0; w < nwg; ++w) t += r[w];
        return t;
    }
    if (wig == 0) {
        float t = lane < nwg ? r[lane] : 0.0f;
        t = warp_sum(t);
        if (lane == 0) r[32] = t;
    }
    __syncthreads();
    return r[32];
}

// Adds each thread's dgamma partial sums (dg[k], column col(k)) to dgamma:
// with one row per block straight from registers, 16-byte reductions where
// dgamma is 16-byte aligned; with several rows per block the groups first add
// theirs in the shared array dgs (H floats), then the block adds dgs once, so
// global additions number about blocks x H / 4.  Called by every thread of
// the block.
template <int V, int NV, class ColFn>
__device__ __forceinline__ void add_dgamma(float *dgamma, int H, int G, const float (&dg)[NV * V], ColFn col_of,
                                           float *dgs)
{
    const bool v4 = (reinterpret_cast<uintptr_t>(dgamma) & 15) == 0;
    if (G == 1) {
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int col = col_of(k);
            if constexpr (V >= 4) {
#pragma unroll
                for (int i = 0; i < V; i += 4)
                    if (col + i < H) {
                        if (v4)
                            red_add_v4(dgamma + col + i, dg[k * V + i], dg[k * V + i + 1], dg[k * V + i + 2],
                                       dg[k * V + i + 3]);
                        else
                            for (int q = 0; q < 4; ++q) atomicAdd(dgamma + col + i + q, dg[k * V + i + q]);
                    }
            } else {
#pragma unroll
                for (int i = 0; i < V; ++i)
                    if (col + i < H) atomicAdd(dgamma + col + i, dg[k * V + i]);
            }
        }
        return;
    }
    for (int j = threadIdx.x; j < H; j += blockDim.x) dgs[j] = 0.0f;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int col = col_of(k);
#pragma unroll
        for (int i = 0; i < V; ++i)
            if (col + i < H) atomicAdd(dgs + col + i, dg[k * V + i]);
    }
    __syncthreads();
    for (int j = threadIdx.x * 4; j < H; j += blockDim.x * 4) {
        if (v4 && j + 4 <= H)
            red_add_v4(dgamma + j, dgs[j], dgs[j + 1], dgs[j + 2], dgs[j + 3]);
        else
            for (int q = 0; q < 4 && j + q < H; ++q) atomicAdd(dgamma + j + q, dgs[j + q]);
    }
}

// ds = rstd * gamma * dy - (rstd^3 / H) * s * sum(gamma * dy * s) (+ dh), written
// to dx (and dres); dgamma accumulates dy * s * rstd.
//
// Rows whose operands are 16-byte aligned and whose inputs are in device
// memory: one persistent block per SM whose threads form `groups` teams of
// `tpr` threads.  A thread owns NV 16-byte columns (the same columns in every
// row, so gamma and the dgamma partial sums stay in registers); a team covers
// a whole row and works on R rows at a time, so every phase of a row (the
// loads, the row sum's warp reduction and team barrier, the gradient) is paid
// once for R rows and has R rows of independent work to overlap.  Element
// pairs use the f32x2 forms.
//
// A stage (teams x R rows of dy, h and dh, and the rows' rstd values) reaches
// a ring of `stages` shared-memory stages through the bulk-copy engine
// (cp.async.bulk, one copy per row and operand; rstd by 4-byte cp.async), all
// completing on the stage's `full` mbarrier, so the loads in flight per SM are
// the ring and not what registers can hold.  Issuing a stage's copies holds
// the issuing warp for about a thousand cycles, so who issues them matters:
//   - PROD (rows of up to 1024 vectors): a producer warp, the block's last,
//     issues every stage once all 8 consumer warps have arrived on the stage's
//     `empty` mbarrier; consumers never issue.  R = 8 / NV rows per team.
//   - otherwise (wider rows, NV = 4 at 512 threads, whose 16 warps leave no
//     registers for a producer warp): each warp counts itself out of a stage
//     when it has read it (a per-stage counter that only grows), and the warp
//     whose count completes the stage refills it.  R = 4 / NV.
// Rows are read from shared memory twice: the first pass forms d * s once for
// the row sum sum(gamma * (d * s)) and the dgamma partial sums, the second
// writes ds.  Teams never wait for one another: a row sum is a warp reduction
// and, for teams of several warps, one named barrier per R rows (the team's
// own) after which every warp reduces the team's warp sums itself.  Waiting
// warps sleep in mbarrier try_wait instead of spinning.
//
// Every wait is bounded (about a second).  A warp whose wait runs out makes
// its whole team stop (the decision is taken at the team's barrier, so it is
// the same for all its warps); a stage that team no longer releases is never
// refilled, so the other teams and the producer run out of waits in turn.  The
// block then waits (bounded) for the copies it issued, counts one timeout and
// leaves dgamma untouched.
constexpr int kRmsBwdConsumersP = 256;      // consumer threads beside the producer warp
constexpr int kRmsBwdThreads = 512;         // threads of the block without one

// Two fp32 lanes per instruction (the f32x2 forms of sm_100 and later); each
// lane is the same IEEE operation, rounded to nearest, as the scalar one.
struct F2 {
    float x, y;
};

__device__ __forceinline__ F2 mul2(F2 a, F2 b)
{
    F2 d;
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ F2 fma2(F2 a, F2 b, F2 c)
{
    F2 d;
    asm("{\n\t.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
        "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ F2 add2(F2 a, F2 b)
{
    F2 d;
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// Element pair q of a 16-byte access (its four words), and back.
template <class C>
__device__ __forceinline__ F2 get_pair(const uint32_t (&w)[4], int q)
{
    if constexpr (C::kPerWord == 2) return F2{C::get(w[q], 0), C::get(w[q], 1)};
    else return F2{C::get(w[2 * q], 0), C::get(w[2 * q + 1], 0)};
}

template <class C>
__device__ __forceinline__ void put_pair(uint32_t (&w)[4], int q, F2 v)
{
    if constexpr (C::kPerWord == 2) {
        const float f[2] = {v.x, v.y};
        w[q] = C::put(f);
    } else {
        w[2 * q] = C::put(&v.x);
        w[2 * q + 1] = C::put(&v.y);
    }
}

template <class T, bool DH, int NV, bool PROD>
__global__ void __launch_bounds__(PROD ? kRmsBwdConsumersP + 32 : kRmsBwdThreads, 1)
    add_rmsnorm_bwd_staged_kernel(const BwdParams p)
{
    using C = Codec<T>;
    constexpr int V = 16 / int(sizeof(T));      // elements per 16-byte access
    constexpr int QV = V / 2;                   // element pairs per access
    constexpr int R = (PROD ? 8 : 4) / NV;      // rows per team per stage
    constexpr int W = 4;
    constexpr int nin = DH ? 3 : 2;
    extern __shared__ __align__(128) unsigned char smem[];
    const int TM = p.groups, tpr = p.tpr, S = p.stages;
    const int SR = TM * R;                      // rows per stage
    const int consumers = TM * tpr;
    const int warps = consumers >> 5, nwg = tpr >> 5;
    const uint32_t rb = uint32_t(p.H) * uint32_t(sizeof(T));        // one operand row, bytes
    const uint32_t stage_bytes = uint32_t(SR * nin) * rb;           // layout [operand][stage row][H]
    unsigned char *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + size_t(S) * stage_bytes);
    uint64_t *empty = full + S;                                     // PROD: [S] consumer warps done
    int *last_issued = reinterpret_cast<int *>(full + S);           // otherwise: [S], then
    int *done = last_issued + S;                                    //   [S] warps counted out, ever
    float *rss = reinterpret_cast<float *>(full + 2 * S);           // [S][SR] rstd of the staged rows
    float *red = rss + S * SR;                                      // [2][SR][nwg] warp sums
    volatile int *gabort = reinterpret_cast<volatile int *>(red + 2 * SR * nwg);   // [2][TM]

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            if constexpr (PROD) {
                mbar_init(smem_u32(&empty[s]), uint32_t(warps));
            } else {
                last_issued[s] = -1;
                done[s] = 0;
            }
        }
        for (int i = 0; i < 2 * TM; ++i) gabort[i] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    // the block's first stage of rows (dy, h and dh), asked of L2 before the wait
    if (warp == 0) {
        const int64_t base = int64_t(blockIdx.x) * SR;
        const int n = base < p.rows ? int(p.rows - base < SR ? p.rows - base : SR) : 0;
        for (int j = lane; j < n * nin; j += 32) {
            const int op = j / n, r = j - op * n;
            const char *src = op == 0   ? p.dy + (base + r) * p.sdy
                              : op == 1 ? p.h + (base + r) * p.sh
                                        : p.dh + (base + r) * p.sdh;
            prefetch_bulk(src, rb);
        }
    }
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // iterations per block fit 32 bits: rows of at least 16 bytes in device memory number below 2^35
    const int64_t n_stages = (p.rows + SR - 1) / SR;
    const int iters = n_stages > blockIdx.x ? int((n_stages - 1 - blockIdx.x) / gridDim.x + 1) : 0;
    // a whole warp: the copies of iteration `it` into stage it % S
    const auto issue = [&](int it) {
        const int64_t base = (int64_t(blockIdx.x) + int64_t(it) * gridDim.x) * SR;
        const int n = int(p.rows - base < SR ? p.rows - base : SR);
        const int s = it % S;
        const uint32_t bar = smem_u32(&full[s]);
        const uint32_t dst = smem_u32(ring + size_t(s) * stage_bytes);
        // the rstd copies join the phase before the arrival that can end it
        if (lane < n) {
            for (int r = lane; r < n; r += 32) cp_async4(smem_u32(rss + s * SR + r), p.rstd + base + r);
            cp_async_arrive(bar);
        }
        __syncwarp();
        if (lane == 0) {
            if constexpr (!PROD) last_issued[s] = it;
            mbar_expect_tx(bar, uint32_t(n * nin) * rb);
        }
        __syncwarp();
        for (int j = lane; j < n * nin; j += 32) {
            const int op = j / n, r = j - op * n;
            const char *src = op == 0   ? p.dy + (base + r) * p.sdy
                              : op == 1 ? p.h + (base + r) * p.sh
                                        : p.dh + (base + r) * p.sdh;
            bulk_load(dst + uint32_t(op * SR + r) * rb, src, rb, bar);
        }
    };

    const int t = threadIdx.x / tpr, tg = threadIdx.x - t * tpr;     // team, thread within the team
    const auto column = [&](int k) { return (tg + k * tpr) * V; };
    F2 dg[NV * QV];
#pragma unroll
    for (int i = 0; i < NV * QV; ++i) dg[i] = F2{0.0f, 0.0f};
    bool failed = false;

    if (PROD && threadIdx.x >= consumers) {
        // the producer warp: stage it % S is filled for the (it / S)-th time
        int it = 0;
        for (; it < iters; ++it) {
            if (it >= S) {
                bool ok = true;
                if (lane == 0) ok = mbar_wait_sleep(smem_u32(&empty[it % S]), uint32_t((it / S - 1) & 1));
                if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) {
                    failed = true;
                    break;
                }
            }
            issue(it);
        }
        // the block may only end once every copy it issued has landed
        bool ok = true;
        if (lane == 0)
            for (int j = it > S ? it - S : 0; j < it && ok; ++j)
                ok = mbar_wait_sleep(smem_u32(&full[j % S]), uint32_t((j / S) & 1));
        if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) failed = true;
    } else {
        if (!PROD && warp == 0)
            for (int it = 0; it < S && it < iters; ++it) issue(it);
        const int wig = tg >> 5;
        uint32_t gw[NV][W];
#pragma unroll
        for (int k = 0; k < NV; ++k)
            if (column(k) < p.H) Access<16>::load(p.gamma + int64_t(column(k)) * sizeof(T), gw[k]);

        for (int it = 0; it < iters; ++it) {
            const int s = it % S, par = it & 1;
            const int64_t row0 = (int64_t(blockIdx.x) + int64_t(it) * gridDim.x) * SR + t * R;
            const bool landed =
                __all_sync(0xFFFFFFFFu, mbar_wait_sleep(smem_u32(&full[s]), uint32_t((it / S) & 1)));
            const unsigned char *st = ring + size_t(s) * stage_bytes + size_t(t * R) * rb;
            const size_t op_stride = size_t(SR) * rb;
            float rs[R];
            F2 dot[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                rs[r] = landed && row0 + r < p.rows ? rss[s * SR + t * R + r] : 0.0f;
                dot[r] = F2{0.0f, 0.0f};
            }
            if (landed) {
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    const int col = column(k);
                    if (col < p.H) {
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            if (row0 + r < p.rows) {
                                const unsigned char *q0 = st + size_t(r) * rb + size_t(col) * sizeof(T);
                                const uint4 d4 = *reinterpret_cast<const uint4 *>(q0);
                                const uint4 s4 = *reinterpret_cast<const uint4 *>(q0 + op_stride);
                                const uint32_t wd[W] = {d4.x, d4.y, d4.z, d4.w}, ws[W] = {s4.x, s4.y, s4.z, s4.w};
                                const F2 rs2{rs[r], rs[r]};
#pragma unroll
                                for (int q = 0; q < QV; ++q) {
                                    const F2 ds = mul2(get_pair<C>(wd, q), get_pair<C>(ws, q));
                                    dg[k * QV + q] = fma2(ds, rs2, dg[k * QV + q]);
                                    dot[r] = fma2(get_pair<C>(gw[k], q), ds, dot[r]);
                                }
                            }
                        }
                    }
                }
            }
            float tot[R];
#pragma unroll
            for (int r = 0; r < R; ++r) tot[r] = warp_sum(dot[r].x + dot[r].y);
            bool go = landed;
            if (nwg > 1) {
                float *rr = red + (par * SR + t * R) * nwg;
                if (lane == 0) {
#pragma unroll
                    for (int r = 0; r < R; ++r) rr[r * nwg + wig] = tot[r];
                    if (!landed) gabort[par * TM + t] = 1;
                }
                named_barrier(1 + t, tpr);
                go = gabort[par * TM + t] == 0;
#pragma unroll
                for (int r = 0; r < R; ++r) tot[r] = warp_sum(lane < nwg ? rr[r * nwg + lane] : 0.0f);
            }
            if (!go) {
                failed = true;
                break;
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (row0 + r < p.rows) {
                    const float c = rs[r] * rs[r] * rs[r] * (tot[r] / float(p.H));
                    const F2 nc2{-c, -c}, rs2{rs[r], rs[r]};
                    char *dxr = p.dx + (row0 + r) * p.sdx, *drr = p.dres ? p.dres + (row0 + r) * p.sdr : nullptr;
#pragma unroll
                    for (int k = 0; k < NV; ++k) {
                        const int col = column(k);
                        if (col < p.H) {
                            const unsigned char *q0 = st + size_t(r) * rb + size_t(col) * sizeof(T);
                            const uint4 d4 = *reinterpret_cast<const uint4 *>(q0);
                            const uint4 s4 = *reinterpret_cast<const uint4 *>(q0 + op_stride);
                            const uint32_t wd[W] = {d4.x, d4.y, d4.z, d4.w}, ws[W] = {s4.x, s4.y, s4.z, s4.w};
                            uint32_t we[W] = {0, 0, 0, 0};
                            if constexpr (DH) {
                                const uint4 e4 = *reinterpret_cast<const uint4 *>(q0 + 2 * op_stride);
                                we[0] = e4.x, we[1] = e4.y, we[2] = e4.z, we[3] = e4.w;
                            }
                            uint32_t wo[W];
#pragma unroll
                            for (int q = 0; q < QV; ++q) {
                                // rs * gamma * d - c * s (+ dh)
                                const F2 tq = mul2(mul2(rs2, get_pair<C>(gw[k], q)), get_pair<C>(wd, q));
                                F2 f = fma2(nc2, get_pair<C>(ws, q), tq);
                                if constexpr (DH) f = add2(f, get_pair<C>(we, q));
                                put_pair<C>(wo, q, f);
                            }
                            const int64_t off = int64_t(col) * sizeof(T);
                            Access<16>::store(dxr + off, wo);
                            if (drr) Access<16>::store(drr + off, wo);
                        }
                    }
                }
            }
            __syncwarp();
            if constexpr (PROD) {
                // this warp is done with stage s
                if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
            } else {
                // count this warp out of stage s; the warp that completes the count refills it
                int last = 0;
                if (lane == 0) {
                    __threadfence_block();      // this warp's reads of the stage before its count
                    last = (atomicAdd(&done[s], 1) + 1) % warps == 0;
                    if (last) __threadfence_block();   // every other warp's count before the refill
                }
                if (__shfl_sync(0xFFFFFFFFu, last, 0) && it + S < iters) issue(it + S);
            }
        }
    }
    if (__syncthreads_or(failed)) {
        if (threadIdx.x == 0) {
            atomicAdd(&g_rms_timeouts, 1u);
            // the block may only end once every copy it issued has landed (the
            // producer warp has already waited for its own)
            if constexpr (!PROD) {
                for (int s = 0; s < S; ++s) {
                    const int j = last_issued[s];
                    if (j >= 0 && !mbar_wait_sleep(smem_u32(&full[s]), uint32_t((j / S) & 1))) break;
                }
            }
        }
        return;
    }
    if (!p.dgamma) return;
    float dgf[NV * V];
#pragma unroll
    for (int i = 0; i < NV * QV; ++i) dgf[2 * i] = dg[i].x, dgf[2 * i + 1] = dg[i].y;
    // every copy has landed and been read: the ring is free for the team sums
    // (a producer warp's partial sums are zero)
    add_dgamma<V, NV>(p.dgamma, p.H, TM, dgf, column, reinterpret_cast<float *>(ring));
}

// Narrow 16-byte rows (up to 128 vectors, 1024 elements of 16-bit types):
// the persistent staged kernel would give each block fewer than two stages,
// so its fill and drain, and a launch the next one cannot overlap, decide the
// time.  This kernel is not persistent: a block of 256 threads takes 4 rows
// for each of its teams (one 16-byte access per operand per thread), loads
// them straight into registers, forms the row sums (a warp reduction and the
// team's named barrier), writes ds from the same registers and adds the
// block's dgamma partial sums once, with 16-byte reductions.  A block holds
// 4.2 KiB of shared memory and at most 128 registers a thread: two per SM.
constexpr int kRmsBwdNarrowThreads = 256;
constexpr int kRmsBwdNarrowRows = 4;        // rows per team

template <class T, bool DH>
__global__ void __launch_bounds__(kRmsBwdNarrowThreads, 2)
    add_rmsnorm_bwd_narrow_kernel(const BwdParams p)
{
    using C = Codec<T>;
    constexpr int V = 16 / int(sizeof(T));      // elements per 16-byte access
    constexpr int QV = V / 2;                   // element pairs per access
    constexpr int R = kRmsBwdNarrowRows;
    constexpr int W = 4;
    __shared__ float red[kRmsBwdNarrowThreads / 32 * R];          // [team][R][warps of the team]: 32
    __shared__ float dgs[1024];                                   // the teams' dgamma partial sums
    const int TM = p.groups, tpr = p.tpr, nwg = tpr >> 5;

    const int lane = threadIdx.x & 31;
    const int t = threadIdx.x / tpr, tg = threadIdx.x - t * tpr, wig = tg >> 5;
    const int col = tg * V;
    const bool on_col = t < TM && col < p.H;
    const int64_t row0 = (int64_t(blockIdx.x) * TM + t) * R;

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // the team's rows of dy and h, asked of L2 before the wait
    if (t < TM && tg < R) {
        const int64_t row = row0 + tg;
        if (row < p.rows) {
            prefetch_bulk(p.dy + row * p.sdy, uint32_t(p.H) * sizeof(T));
            prefetch_bulk(p.h + row * p.sh, uint32_t(p.H) * sizeof(T));
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");

    uint32_t gw[W] = {0, 0, 0, 0};
    if (on_col) Access<16>::load(p.gamma + int64_t(col) * sizeof(T), gw);
    // every row of this thread's team, loaded before any arithmetic
    uint32_t wd[R][W], ws[R][W];
    float rs[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t row = row0 + r;
        const bool on = on_col && row < p.rows;
        rs[r] = on ? p.rstd[row] : 0.0f;
        if (on) {
            Access<16>::load(p.dy + row * p.sdy + int64_t(col) * sizeof(T), wd[r]);
            Access<16>::load(p.h + row * p.sh + int64_t(col) * sizeof(T), ws[r]);
        } else {
#pragma unroll
            for (int j = 0; j < W; ++j) wd[r][j] = ws[r][j] = 0;
        }
    }
    F2 dg[QV];
#pragma unroll
    for (int q = 0; q < QV; ++q) dg[q] = F2{0.0f, 0.0f};
    float tot[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        F2 dot{0.0f, 0.0f};
        const F2 rs2{rs[r], rs[r]};
#pragma unroll
        for (int q = 0; q < QV; ++q) {
            const F2 ds = mul2(get_pair<C>(wd[r], q), get_pair<C>(ws[r], q));
            dg[q] = fma2(ds, rs2, dg[q]);
            dot = fma2(get_pair<C>(gw, q), ds, dot);
        }
        tot[r] = warp_sum(dot.x + dot.y);
    }
    if (nwg > 1) {
        float *rr = red + t * R * nwg;
        if (lane == 0 && t < TM) {
#pragma unroll
            for (int r = 0; r < R; ++r) rr[r * nwg + wig] = tot[r];
        }
        if (t < TM) named_barrier(1 + t, tpr);
#pragma unroll
        for (int r = 0; r < R; ++r) tot[r] = warp_sum(lane < nwg && t < TM ? rr[r * nwg + lane] : 0.0f);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t row = row0 + r;
        if (!on_col || row >= p.rows) continue;
        const float c = rs[r] * rs[r] * rs[r] * (tot[r] / float(p.H));
        const F2 nc2{-c, -c}, rs2{rs[r], rs[r]};
        uint32_t we[W] = {0, 0, 0, 0};
        if constexpr (DH) Access<16>::load(p.dh + row * p.sdh + int64_t(col) * sizeof(T), we);
        uint32_t wo[W];
#pragma unroll
        for (int q = 0; q < QV; ++q) {
            // rs * gamma * d - c * s (+ dh)
            const F2 tq = mul2(mul2(rs2, get_pair<C>(gw, q)), get_pair<C>(wd[r], q));
            F2 f = fma2(nc2, get_pair<C>(ws[r], q), tq);
            if constexpr (DH) f = add2(f, get_pair<C>(we, q));
            put_pair<C>(wo, q, f);
        }
        const int64_t off = int64_t(col) * sizeof(T);
        Access<16>::store(p.dx + row * p.sdx + off, wo);
        if (p.dres) Access<16>::store(p.dres + row * p.sdr + off, wo);
    }
    if (!p.dgamma) return;
    float dgf[V];
#pragma unroll
    for (int q = 0; q < QV; ++q) dgf[2 * q] = dg[q].x, dgf[2 * q + 1] = dg[q].y;
    // threads outside every team hold zeros; their columns are valid ones
    add_dgamma<V, 1>(p.dgamma, p.H, TM, dgf, [&](int) { return on_col ? col : 0; }, dgs);
}

// Rows of up to 512 16-byte vectors of 16-bit types (4096 elements) or 384 of
// fp32 (1536 elements) in device memory, where the staged kernel's ring would
// hold only a few stages per SM and its fill and drain would decide the time:
// a persistent grid of register teams.
//   - One block per SM of up to 1024 threads (64 registers each) holds G teams
//     of tpr threads.  A team works on one row at a time and a thread on NV
//     16-byte vectors of it (vector k * tpr + tg), loaded straight into
//     registers before any arithmetic, so an SM keeps up to 1024 x NV x 32
//     bytes of dy and h in flight.
//   - Rows go to the teams round robin over the blocks (row (i * G + t) * grid
//     + block), which spreads them evenly over the SMs.  Before waiting for the
//     previous grid a team asks L2 for its first row; each row's loads come with
//     an L2 prefetch of the team's next row.
//   - gamma sits in shared memory.  Each team adds its dgamma partial sums to a
//     private fp32 row in shared memory (each element read, added and written
//     back by the thread that owns its column; the two halves of a 16-bit
//     vector's eight columns lie in two half-rows, so a warp's 16-byte accesses
//     do not collide in the banks), and the block adds the sum of its teams'
//     rows to dgamma once at the end.
//   - A team of several warps shares its warp sums through shared memory under
//     its own named barrier (at most 15 teams then); consecutive rows alternate
//     between two exchange arrays, as in group_sum.
constexpr int kRmsBwdTeamThreads = 1024;

// The team kernel's final dgamma sum: P threads per group of four columns
// (a power of two, at most 8 and at most the teams), and the stride in floats
// of the teams' shared-memory rows, padded so that the 16-byte reads of the
// P threads (rows u, u + 1, ...) and of their neighbours fall in distinct banks.
__host__ __device__ inline int team_parts(int H, int threads, int G)
{
    int P = 1;
    while (P < 8 && P < G && (H / 4) * (2 * P) <= threads) P *= 2;
    return P;
}

__host__ __device__ inline int team_stride(int H, int P)
{
    return P == 1 ? H : (H + 31) / 32 * 32 + 32 / P;
}

// An L2 prefetch of the 128-byte line that holds q, issued only by the thread
// whose 16-byte vector starts the line.
__device__ __forceinline__ void prefetch_line(const char *q)
{
    if ((reinterpret_cast<uintptr_t>(q) & 127) < 16) asm volatile("prefetch.global.L2 [%0];" ::"l"(q));
}

template <class T, bool DH, int NV>
__global__ void __launch_bounds__(kRmsBwdTeamThreads, 1)
    add_rmsnorm_bwd_teams_kernel(const BwdParams p)
{
    using C = Codec<T>;
    constexpr int V = 16 / int(sizeof(T));      // elements per 16-byte access
    constexpr int QV = V / 2;                   // element pairs per access
    extern __shared__ __align__(16) unsigned char team_smem[];
    const int G = p.groups, tpr = p.tpr, H = p.H, nvec = H / V, nwg = tpr >> 5;
    const int P = team_parts(H, blockDim.x, G), Hp = team_stride(H, P);
    // [nvec] 16-byte gamma vectors, then [G][Hp] dgamma partial sums, then
    // [2][G][nwg] warp sums; H * sizeof(T) and Hp * 4 are multiples of 16
    const char *gsm = reinterpret_cast<const char *>(team_smem);
    float *dgs = reinterpret_cast<float *>(team_smem + int64_t(nvec) * 16);
    float *xch = dgs + int64_t(G) * Hp;

    const int t = threadIdx.x / tpr, tg = threadIdx.x - t * tpr, lane = threadIdx.x & 31, wig = tg >> 5;
    const int64_t step = int64_t(gridDim.x) * G;
    int64_t row = int64_t(t) * gridDim.x + blockIdx.x;

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // Before waiting for the previous grid, ask L2 for the team's first row of
    // dy and h, so that DRAM starts on it during that grid's last blocks.  L2 is
    // the point of coherence: a line the previous grid writes after the
    // prefetch is simply fetched again, and nothing is read from the core's
    // own caches before the wait.
    if (row < p.rows) {
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int jv = k * tpr + tg;
            if (jv < nvec) {
                const int64_t off = int64_t(jv) * 16;
                prefetch_line(p.dy + row * p.sdy + off);
                prefetch_line(p.h + row * p.sh + off);
            }
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    uint32_t wd[NV][4], ws[NV][4], we[DH ? NV : 1][4];
    float rs = 0.0f;
    // a row's loads, and an L2 prefetch of the team's next row
    const auto load_row = [&](int64_t r) {
        rs = p.rstd[r];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int jv = k * tpr + tg;
            if (jv < nvec) {
                const int64_t off = int64_t(jv) * 16;
                Access<16>::load(p.dy + r * p.sdy + off, wd[k]);
                Access<16>::load(p.h + r * p.sh + off, ws[k]);
                if constexpr (DH) Access<16>::load(p.dh + r * p.sdh + off, we[k]);
            }
        }
        if (r + step < p.rows) {
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int jv = k * tpr + tg;
                if (jv < nvec) {
                    const int64_t off = int64_t(jv) * 16;
                    prefetch_line(p.dy + (r + step) * p.sdy + off);
                    prefetch_line(p.h + (r + step) * p.sh + off);
                }
            }
        }
    };
    // the first row's loads go out before gamma is staged
    if (row < p.rows) load_row(row);
    for (int j = threadIdx.x; j < nvec; j += blockDim.x) {
        uint32_t w[4];
        Access<16>::load(p.gamma + int64_t(j) * 16, w);
        *reinterpret_cast<uint4 *>(team_smem + int64_t(j) * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncthreads();

    float *mydg = dgs + int64_t(t) * Hp;
    const int half = V == 8 ? H / 2 : 0;        // offset of a 16-bit vector's upper four columns
    const auto gamma_vec = [&](int jv, uint32_t (&w)[4]) {
        const uint4 g = *reinterpret_cast<const uint4 *>(gsm + int64_t(jv) * 16);
        w[0] = g.x, w[1] = g.y, w[2] = g.z, w[3] = g.w;
    };
    int parity = 0;
    for (bool first = true; row < p.rows; first = false, parity ^= 1) {
        // row sum of gamma * (dy * s); dgamma partial sums dy * s * rstd (the
        // team's first row writes its shared-memory row, later rows add to it)
        F2 dot{0.0f, 0.0f};
        const F2 rs2{rs, rs};
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int jv = k * tpr + tg;
            if (jv >= nvec) continue;
            uint32_t gw[4];
            gamma_vec(jv, gw);
            float4 *dst[2] = {reinterpret_cast<float4 *>(mydg + jv * 4),
                              reinterpret_cast<float4 *>(mydg + half + jv * 4)};
            float4 a[2] = {make_float4(0.0f, 0.0f, 0.0f, 0.0f), make_float4(0.0f, 0.0f, 0.0f, 0.0f)};
            if (!first) {
                a[0] = *dst[0];
                if constexpr (V == 8) a[1] = *dst[1];
            }
#pragma unroll
            for (int q = 0; q < QV; ++q) {
                const F2 ds = mul2(get_pair<C>(wd[k], q), get_pair<C>(ws[k], q));
                dot = fma2(get_pair<C>(gw, q), ds, dot);
                float4 &acc = a[q / 2];
                F2 cur = (q & 1) ? F2{acc.z, acc.w} : F2{acc.x, acc.y};
                cur = fma2(ds, rs2, cur);
                if (q & 1) acc.z = cur.x, acc.w = cur.y;
                else acc.x = cur.x, acc.y = cur.y;
            }
            *dst[0] = a[0];
            if constexpr (V == 8) *dst[1] = a[1];
        }
        float tot = warp_sum(dot.x + dot.y);
        if (nwg > 1) {
            float *r = xch + (parity * G + t) * nwg;
            if (lane == 0) r[wig] = tot;
            named_barrier(1 + t, tpr);
            tot = 0.0f;
            for (int w = 0; w < nwg; ++w) tot += r[w];
        }
        const float c = rs * rs * rs * (tot / float(H));
        const F2 nc2{-c, -c};
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int jv = k * tpr + tg;
            if (jv >= nvec) continue;
            uint32_t gw[4], wo[4];
            gamma_vec(jv, gw);
#pragma unroll
            for (int q = 0; q < QV; ++q) {
                // rs * gamma * d - c * s (+ dh)
                const F2 tq = mul2(mul2(rs2, get_pair<C>(gw, q)), get_pair<C>(wd[k], q));
                F2 f = fma2(nc2, get_pair<C>(ws[k], q), tq);
                if constexpr (DH) f = add2(f, get_pair<C>(we[k], q));
                put_pair<C>(wo, q, f);
            }
            const int64_t off = int64_t(jv) * 16;
            Access<16>::store(p.dx + row * p.sdx + off, wo);
            if (p.dres) Access<16>::store(p.dres + row * p.sdr + off, wo);
        }
        row += step;
        if (row < p.rows) load_row(row);
    }
    if (!p.dgamma) return;
    __syncthreads();
    // The block's sum over the teams that had a row (team u: u * grid + block <
    // rows), four columns at a time.  P consecutive threads share a group of
    // four columns, each adding every P-th team, and combine by shuffles.
    const int quads = H / 4;
    const int64_t rem = p.rows - blockIdx.x, reach = (rem + gridDim.x - 1) / gridDim.x;
    const int had = rem <= 0 ? 0 : reach < G ? int(reach) : G;     // teams of this block with a row
    const bool v4 = (reinterpret_cast<uintptr_t>(p.dgamma) & 15) == 0;
    for (int base = 0; base < quads * P; base += blockDim.x) {
        const int idx = base + threadIdx.x, qd = idx / P, part = idx - qd * P;
        float4 s = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (qd < quads) {
            const int j = qd * 4, jv = j / V, i0 = j - jv * V;
            const float *src = dgs + (i0 >= 4 ? half : 0) + jv * 4;
            for (int u = part; u < had; u += P) {
                const float4 v = *reinterpret_cast<const float4 *>(src + int64_t(u) * Hp);
                s.x += v.x, s.y += v.y, s.z += v.z, s.w += v.w;
            }
        }
        for (int o = 1; o < P; o *= 2) {
            s.x += __shfl_xor_sync(0xFFFFFFFFu, s.x, o);
            s.y += __shfl_xor_sync(0xFFFFFFFFu, s.y, o);
            s.z += __shfl_xor_sync(0xFFFFFFFFu, s.z, o);
            s.w += __shfl_xor_sync(0xFFFFFFFFu, s.w, o);
        }
        if (qd < quads && part == 0 && had > 0) {
            float *d = p.dgamma + qd * 4;
            if (v4) {
                red_add_v4(d, s.x, s.y, s.z, s.w);
            } else {
                atomicAdd(d, s.x);
                atomicAdd(d + 1, s.y);
                atomicAdd(d + 2, s.z);
                atomicAdd(d + 3, s.w);
            }
        }
    }
}

// Rows that are not 16-byte aligned: the same arithmetic with element
// accesses, each thread owning EPT columns t + k * tpr, one load of each
// element per pass (the second pass's loads hit the cache).
template <class T, int EPT>
__global__ void __launch_bounds__(1024)
    add_rmsnorm_bwd_kernel(const BwdParams p)
{
    using C = Codec<T>;
    extern __shared__ float dsm[];      // [2][groups][33] row sums, then H floats of dgamma (groups > 1)
    const int G = p.groups, tpr = p.tpr;

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const int g = threadIdx.x / tpr, tg = threadIdx.x - g * tpr;
    const int lane = threadIdx.x & 31, wig = tg >> 5, nwg = tpr >> 5;
    const auto column = [&](int k) { return tg + k * tpr; };
    // gamma is read where it is used (it stays in L1): keeping it in registers
    // beside the dgamma partial sums would spill at 1024 threads
    const auto gam = [&](int col) { return C::load1(p.gamma + int64_t(col) * sizeof(T)); };
    float dg[EPT];
#pragma unroll
    for (int k = 0; k < EPT; ++k) dg[k] = 0.0f;

    int parity = 0;
    for (int64_t base = int64_t(blockIdx.x) * G; base < p.rows; base += int64_t(gridDim.x) * G, parity ^= 1) {
        const int64_t row = base + g;
        const bool on = row < p.rows;
        const float rs = on ? p.rstd[row] : 0.0f;
        const char *dyr = p.dy + row * p.sdy, *hr = p.h + row * p.sh;
        const char *dhr = p.dh ? p.dh + row * p.sdh : nullptr;
        char *dxr = p.dx + row * p.sdx, *drr = p.dres ? p.dres + row * p.sdr : nullptr;
        SumSq<EPT> dot;
#pragma unroll
        for (int k = 0; k < EPT; ++k) {
            const int col = column(k);
            if (on && col < p.H) {
                const int64_t off = int64_t(col) * sizeof(T);
                dot.add(k, gam(col), C::load1(dyr + off) * C::load1(hr + off));
            }
        }
        const float c = rs * rs * rs * (group_sum(dot.total(), dsm + (parity * G + g) * 33, lane, wig, nwg) /
                                        float(p.H));
#pragma unroll
        for (int k = 0; k < EPT; ++k) {
            const int col = column(k);
            if (on && col < p.H) {
                const int64_t off = int64_t(col) * sizeof(T);
                const float d = C::load1(dyr + off), sv = C::load1(hr + off);
                float v = rs * gam(col) * d - c * sv;
                if (dhr) v += C::load1(dhr + off);
                dg[k] = fmaf(d * sv, rs, dg[k]);
                C::store1(dxr + off, v);
                if (drr) C::store1(drr + off, v);
            }
        }
    }
    if (!p.dgamma) return;
    add_dgamma<1, EPT>(p.dgamma, p.H, G, dg, column, dsm + 2 * G * 33);
}

using BwdFn = void (*)(BwdParams);

template <class T, bool DH>
BwdFn pick_staged(int nv, bool prod)
{
    if (!prod) return add_rmsnorm_bwd_staged_kernel<T, DH, 4, false>;
    return nv == 1   ? add_rmsnorm_bwd_staged_kernel<T, DH, 1, true>
           : nv == 2 ? add_rmsnorm_bwd_staged_kernel<T, DH, 2, true>
                     : add_rmsnorm_bwd_staged_kernel<T, DH, 4, true>;
}

// nv = 0: the element kernel; 1, 2 or 4: the staged kernel with nv 16-byte
// accesses per operand per thread, with a producer warp (prod) or without
template <class T>
BwdFn pick_bwd_t(int nv, bool dh, bool prod)
{
    if (nv == 0) return add_rmsnorm_bwd_kernel<T, 16>;
    return dh ? pick_staged<T, true>(nv, prod) : pick_staged<T, false>(nv, prod);
}

template <class T>
BwdFn pick_teams_t(int nv, bool dh)
{
    if (dh) return nv == 1 ? add_rmsnorm_bwd_teams_kernel<T, true, 1> : add_rmsnorm_bwd_teams_kernel<T, true, 2>;
    return nv == 1   ? add_rmsnorm_bwd_teams_kernel<T, false, 1>
           : nv == 2 ? add_rmsnorm_bwd_teams_kernel<T, false, 2>
                     : add_rmsnorm_bwd_teams_kernel<T, false, 4>;
}

// the team kernel with nv 16-byte vectors per operand per thread (at most 2 with dh)
BwdFn pick_teams(int dtype, int nv, bool dh)
{
    switch (dtype) {
    case GLU_F32: return pick_teams_t<float>(nv, dh);
    case GLU_F16: return pick_teams_t<__half>(nv, dh);
    default: return pick_teams_t<__nv_bfloat16>(nv, dh);
    }
}

BwdFn pick_narrow(int dtype, bool dh)
{
    switch (dtype) {
    case GLU_F32: return dh ? add_rmsnorm_bwd_narrow_kernel<float, true> : add_rmsnorm_bwd_narrow_kernel<float, false>;
    case GLU_F16:
        return dh ? add_rmsnorm_bwd_narrow_kernel<__half, true> : add_rmsnorm_bwd_narrow_kernel<__half, false>;
    default:
        return dh ? add_rmsnorm_bwd_narrow_kernel<__nv_bfloat16, true>
                  : add_rmsnorm_bwd_narrow_kernel<__nv_bfloat16, false>;
    }
}

// Blocks of the narrow kernel resident on one SM at once (the occupancy
// query, asked once per device, dtype and dh variant; devices numbered 64
// and above are asked on every call).
cudaError_t narrow_resident(int dev, int dtype, bool dh, int *out)
{
    static std::atomic<int> cache[64][6];
    const int key = (dtype == GLU_F32 ? 0 : dtype == GLU_F16 ? 1 : 2) * 2 + (dh ? 1 : 0);
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev][key].load(std::memory_order_relaxed);
        if (c > 0) { *out = c; return cudaSuccess; }
    }
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &n, reinterpret_cast<const void *>(pick_narrow(dtype, dh)), kRmsBwdNarrowThreads, 0);
    if (e != cudaSuccess) return e;
    if (n < 1) n = 1;
    if (dev >= 0 && dev < 64) cache[dev][key].store(n, std::memory_order_relaxed);
    *out = n;
    return cudaSuccess;
}

BwdFn pick_bwd(int dtype, int nv, bool dh, bool prod)
{
    switch (dtype) {
    case GLU_F32: return pick_bwd_t<float>(nv, dh, prod);
    case GLU_F16: return pick_bwd_t<__half>(nv, dh, prod);
    default: return pick_bwd_t<__nv_bfloat16>(nv, dh, prod);
    }
}

cudaError_t timeouts(unsigned int *count, bool reset)
{
    cudaError_t e = cudaMemcpyFromSymbol(count, g_rms_timeouts, sizeof(unsigned int));
    if (e == cudaSuccess && reset) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_rms_timeouts, &zero, sizeof(unsigned int));
    }
    return e;
}

using KernelFn = void (*)(Params);

template <class T>
KernelFn pick_t(int ept, bool vec, bool rows)
{
    if (rows) return add_rmsnorm_rows_kernel<T, 16 / sizeof(T) * 2>;       // 16 (16-bit) or 8 (f32)
    if (vec) return ept == 16 ? add_rmsnorm_kernel<T, 16, true> : add_rmsnorm_kernel<T, 64, true>;
    return ept == 16 ? add_rmsnorm_kernel<T, 16, false> : add_rmsnorm_kernel<T, 64, false>;
}

KernelFn pick(int dtype, int ept, bool vec, bool rows)
{
    switch (dtype) {
    case GLU_F32: return pick_t<float>(ept, vec, rows);
    case GLU_F16: return pick_t<__half>(ept, vec, rows);
    default: return pick_t<__nv_bfloat16>(ept, vec, rows);
    }
}

}  // namespace rms
}  // namespace glu

extern "C" int glu_add_rmsnorm_fwd(const void *x, int64_t x_stride, const void *residual, int64_t res_stride,
                                   const void *gamma, void *h, int64_t h_stride, void *y, int64_t y_stride,
                                   float *rstd, int64_t n_rows, int64_t n_cols, float eps, glu_dtype_t dtype,
                                   glu_stream_t stream)
{
    using namespace glu::rms;
    bool empty = false;
    const int st = glu::validate_add_rmsnorm(x, x_stride, residual, res_stride, gamma, h, h_stride, y, y_stride,
                                             rstd, n_rows, n_cols, eps, dtype, &empty);
    if (st != GLU_OK) return st;
    if (empty) {
        glu::record_launch(glu_launch_info_t{});
        return GLU_OK;
    }
    const int E = dtype == GLU_F32 ? 4 : 2;
    if (n_rows == 1) x_stride = res_stride = h_stride = y_stride = n_cols;
    const auto a16 = [](const void *q) { return uintptr_t(q) % 16 == 0; };
    const bool vec = a16(x) && a16(residual) && a16(gamma) && a16(h) && a16(y) && (n_cols * E) % 16 == 0 &&
                     (x_stride * E) % 16 == 0 && (res_stride * E) % 16 == 0 && (h_stride * E) % 16 == 0 &&
                     (y_stride * E) % 16 == 0;
    // 16-byte rows of 16 KiB or more that fit 1024 threads of two 16-byte
    // accesses per operand (16 elements of 16-bit types, 8 of f32) take the
    // persistent kernel (measured on GB300: 4 % faster at 32 KiB rows, equal at
    // 16 KiB, 1-5 % slower below); otherwise one block per row with 16
    // elements per thread up to 16384 columns (at most 1024 threads), 64
    // beyond (at most 512 threads)
    const bool rows_kernel = vec && n_cols * E >= 16384 && n_cols <= int64_t(1024) * (32 / E);
    const int ept = rows_kernel ? 32 / E : (n_cols <= 16 * 1024 ? 16 : 64);
    int threads = int((n_cols + ept - 1) / ept);
    threads = (threads + 31) / 32 * 32;
    Params p{};
    p.x = static_cast<const char *>(x);
    p.res = static_cast<const char *>(residual);
    p.gamma = static_cast<const char *>(gamma);
    p.h = static_cast<char *>(h);
    p.y = static_cast<char *>(y);
    p.rstd = rstd;
    p.sx = x_stride * E;
    p.sr = res_stride * E;
    p.sh = h_stride * E;
    p.sy = y_stride * E;
    p.rows = n_rows;
    p.H = int(n_cols);
    p.eps = eps;
    // The L2 prefetch before the dependency wait pays where the blocks resident
    // at the start cover most rows: the persistent kernel, and launches of at
    // most 32 MiB of inputs.  With one block per row over several waves, the
    // later blocks would only prefetch the row they load next (measured: 4096
    // rows of 4096 bf16 3 % slower with it, 1024 / 2048 columns 4 / 2 % faster,
    // the persistent kernel at 8192 / 16384 columns 3 / 2 % faster).
    p.prefetch = vec && (rows_kernel || 2 * n_rows * n_cols * E <= (int64_t(32) << 20));
    KernelFn fn = pick(dtype, ept, vec, rows_kernel);
    int64_t blocks = n_rows;
    if (rows_kernel) {      // persistent: as many blocks as fit on the GPU at once
        int dev = 0, sms = 0, per_sm = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reinterpret_cast<const void *>(fn), threads, 0);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return glu::cuda_fail(e);
        }
        const int64_t slots = int64_t(sms) * (per_sm > 0 ? per_sm : 1);
        blocks = n_rows < slots ? n_rows : slots;
    }
    const unsigned grid = unsigned(blocks < int64_t(INT32_MAX) ? blocks : int64_t(INT32_MAX));

    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(unsigned(threads));
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {&p};
    cudaError_t e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(fn), args);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        cfg.attrs = nullptr;
        cfg.numAttrs = 0;
        e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(fn), args);
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return glu::cuda_fail(e);
    }
    glu_launch_info_t info{};
    info.launched = 1;
    info.vec_bytes = vec ? 16 : E;
    info.unroll = ept;
    info.threads = threads;
    info.grid = int32_t(grid);
    info.path = 4;
    info.vector_units = n_rows;
    glu::record_launch(info);
    return GLU_OK;
}

extern "C" int glu_add_rmsnorm_bwd(const void *dy, int64_t dy_stride, const void *h, int64_t h_stride,
                                   const float *rstd, const void *gamma, const void *dh, int64_t dh_stride, void *dx,
                                   int64_t dx_stride, void *dres, int64_t dres_stride, float *dgamma, int64_t n_rows,
                                   int64_t n_cols, glu_dtype_t dtype, glu_stream_t stream)
{
    using namespace glu::rms;
    bool empty = false;
    const int st = glu::validate_add_rmsnorm_bwd(dy, dy_stride, h, h_stride, rstd, gamma, dh, dh_stride, dx,
                                                 dx_stride, dres, dres_stride, dgamma, n_rows, n_cols, dtype, &empty);
    if (st != GLU_OK) return st;
    if (empty) {
        glu::record_launch(glu_launch_info_t{});
        return GLU_OK;
    }
    // dgamma takes atomic reductions: device memory only
    if (dgamma) {
        bool dev_mem = false;
        const cudaError_t pe = glu::on_device(dgamma, &dev_mem);
        if (pe != cudaSuccess) return glu::cuda_fail(pe);
        if (!dev_mem) return GLU_ERR_VALUE;
    }
    const int E = dtype == GLU_F32 ? 4 : 2;
    if (n_rows == 1) dy_stride = h_stride = dh_stride = dx_stride = dres_stride = n_cols;
    const auto a16 = [](const void *q) { return uintptr_t(q) % 16 == 0; };
    const auto s16 = [E](int64_t st_) { return (st_ * E) % 16 == 0; };
    const int V = 16 / E;            // elements per 16-byte access
    const bool vec = a16(dy) && a16(h) && a16(gamma) && a16(dx) && (!dh || a16(dh)) && (!dres || a16(dres)) &&
                     (n_cols * E) % 16 == 0 && s16(dy_stride) && s16(h_stride) && s16(dx_stride) &&
                     (!dh || s16(dh_stride)) && (!dres || s16(dres_stride)) && n_cols <= int64_t(2048) * V;
    // The staged kernel takes 16-byte rows whose inputs are in device memory
    // (the bulk-copy engine and cp.async are given device memory only);
    // anything else, pinned host memory included, takes the element kernel.
    bool staged = vec;
    for (const void *q : {dy, h, dh, static_cast<const void *>(rstd)}) {
        if (!staged || !q) continue;
        bool dev_mem = false;
        const cudaError_t pe = glu::on_device(q, &dev_mem);
        if (pe != cudaSuccess) return glu::cuda_fail(pe);
        staged = dev_mem;
    }
    // 16-byte rows: rows of up to 1024 vectors take the staged kernel with a
    // producer warp and 256 consumer threads, NV (1, 2 or 4) the fewest
    // accesses per operand per thread that keep a row within them; wider rows
    // take it with 512 threads and NV = 4.  Otherwise 16 elements per thread.
    int dev = 0, sms = 0, smem_sm = 0, smem_block = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem_block, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return glu::cuda_fail(e);
    }
    // Rows of up to 128 vectors take the non-persistent narrow kernel instead
    // (4 rows per team, one access per operand per thread) when its grid fits
    // on the GPU at once (the blocks resident per SM, as the occupancy query
    // reports them, times the SMs): every block adds to dgamma, and more blocks
    // than that queue their additions on the same addresses (measured: 262144
    // rows of 64 took 2.5 times the persistent kernel's time).
    const int64_t narrow_tpr = ((n_cols + V - 1) / V + 31) / 32 * 32;
    const int64_t narrow_rows = kRmsBwdNarrowThreads / narrow_tpr * kRmsBwdNarrowRows;
    bool narrow = staged && n_cols <= int64_t(128) * V;
    if (narrow) {
        int resident = 0;
        e = narrow_resident(dev, dtype, dh != nullptr, &resident);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return glu::cuda_fail(e);
        }
        narrow = (n_rows + narrow_rows - 1) / narrow_rows <= int64_t(resident) * sms;
    }
    // Rows that the narrow kernel does not take, of up to 512 vectors (16-bit
    // types) or 384 (f32): the persistent team kernel, with 4 vectors per
    // operand per thread where a row has at least 4 for every lane of a warp
    // (at most 2 with dh, whose rows are held as well), else 2 or 1.
    // (Measured against the staged kernel, both with their first rows asked
    // of L2 before the dependency wait: 1.1-1.4 times faster at 4096 rows of
    // 1024-3072 bf16, 1.06 at 4096 and 1.35 at 1024 x 4096, twice as fast at
    // 65536 rows of 256; 8 % slower at 4096 rows of 2048 f32, 512 vectors.)
    const int64_t nvec = n_cols / V;
    int nvt = 0;
    if (staged && !narrow && nvec <= (E == 2 ? 512 : 384)) {
        nvt = nvec >= 128 ? 4 : nvec >= 64 ? 2 : 1;
        if (dh && nvt > 2) nvt = 2;
    }
    const bool prod = staged && !narrow && !nvt && n_cols <= int64_t(1024) * V;
    const int nv = nvt ? nvt : !staged ? 0 : n_cols <= int64_t(256) * V ? 1 : n_cols <= int64_t(512) * V ? 2 : 4;
    const int ept = staged ? nv * V : 16;
    int tpr = int((n_cols + ept - 1) / ept);
    tpr = (tpr + 31) / 32 * 32;
    // several rows per block for narrow rows, so that fewer blocks add to
    // dgamma: the staged kernel's teams fill its consumer threads (at most 8
    // teams of several warps, one named barrier each, or single-warp teams),
    // the element kernel up to 512 threads
    // (the team kernel: as many teams as 1024 threads hold, at most 15 teams of
    // several warps, which take one named barrier each)
    const int team_threads = narrow ? kRmsBwdNarrowThreads
                             : nvt  ? kRmsBwdTeamThreads
                             : prod ? kRmsBwdConsumersP
                                    : kRmsBwdThreads;
    int groups = tpr >= team_threads ? 1 : (team_threads / tpr < 16 ? team_threads / tpr : 16);
    if (nvt) {
        // then only as many as spread the rows evenly over the SMs: k rows per
        // team at most, the fewest teams per block that take them
        const int64_t gmax = tpr == 32 ? team_threads / 32 : (groups < 15 ? groups : 15);
        const int64_t k = (n_rows + sms * gmax - 1) / (sms * gmax);
        const int64_t need = (n_rows + k - 1) / k, g = (need + sms - 1) / sms;
        groups = int(g < gmax ? g : gmax);
    }
    const int threads = narrow ? kRmsBwdNarrowThreads : tpr * groups + (prod ? 32 : 0);
    const int rows_per_stage = narrow   ? groups * kRmsBwdNarrowRows
                               : nvt    ? groups
                               : staged ? groups * ((prod ? 8 : 4) / nv)
                                        : groups;
    BwdFn fn = narrow ? pick_narrow(dtype, dh != nullptr)
               : nvt  ? pick_teams(dtype, nvt, dh != nullptr)
                      : pick_bwd(dtype, nv, dh != nullptr, prod);

    size_t smem = sizeof(float) * (size_t(2 * groups * 33) + (groups > 1 ? size_t(n_cols) : 0));
    int stages = 0, per_sm = 1;
    if (narrow) {
        smem = 0;       // static shared memory only
    } else if (nvt) {
        // gamma, the teams' dgamma rows and the warp-sum exchange; one block per SM
        const int stride = team_stride(int(n_cols), team_parts(int(n_cols), tpr * groups, groups));
        smem = size_t(nvec) * 16 + sizeof(float) * (size_t(groups) * size_t(stride) + 2 * size_t(groups) * (tpr / 32));
        static std::atomic<int> opted_teams[64][15];
        std::atomic<int> &flag = opted_teams[dev % 64][((dtype == GLU_F32 ? 0 : dtype == GLU_F16 ? 1 : 2) * 5) +
                                                       (dh ? 3 : 0) + (nvt == 4 ? 2 : nvt - 1)];
        if (!flag.load(std::memory_order_acquire)) {
            e = cudaFuncSetAttribute(reinterpret_cast<const void *>(fn), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     smem_block);
            if (e != cudaSuccess) {
                (void)cudaGetLastError();
                return glu::cuda_fail(e);
            }
            flag.store(1, std::memory_order_release);
        }
    } else if (staged) {
        // One block per SM with the deepest ring of stages (dy, h and dh rows,
        // the mbarrier, last issued stage, counter and rstd values) that
        // fits, 8 at most.  A stage holds at most 512 x 64 bytes per operand,
        // 96 KiB for three, so at least 2 fit.
        // per device and kernel: the shared-memory limit raised once
        static std::atomic<int> opted[64][24];
        std::atomic<int> &flag = opted[dev % 64][((dtype == GLU_F32 ? 0 : dtype == GLU_F16 ? 1 : 2) * 2 +
                                                   (dh != nullptr)) * 4 + (prod ? (nv == 4 ? 2 : nv - 1) : 3)];
        if (!flag.load(std::memory_order_acquire)) {
            e = cudaFuncSetAttribute(reinterpret_cast<const void *>(fn), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     smem_block);
            if (e != cudaSuccess) {
                (void)cudaGetLastError();
                return glu::cuda_fail(e);
            }
            flag.store(1, std::memory_order_release);
        }
        const size_t stage = size_t(rows_per_stage) * (dh ? 3 : 2) * size_t(n_cols) * E;
        const size_t per_stage = stage + 16 + size_t(rows_per_stage) * sizeof(float);   // rows, 2 x 8 B, rstd
        const size_t fixed =
            2 * size_t(rows_per_stage) * (tpr / 32) * sizeof(float) + 2 * size_t(groups) * sizeof(int);
        const int64_t room = int64_t(smem_sm) - 1024 < int64_t(smem_block) ? int64_t(smem_sm) - 1024
                                                                              : int64_t(smem_block);
        while (stages < 8 && int64_t((stages + 1) * per_stage + fixed) <= room) ++stages;
        if (stages < 2) return GLU_ERR_SHAPE;     // not reachable within the column limit
        smem = size_t(stages) * per_stage + fixed;
    } else {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reinterpret_cast<const void *>(fn), threads, smem);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return glu::cuda_fail(e);
        }
        if (per_sm < 1) per_sm = 1;
    }
    const int64_t slots = int64_t(sms) * per_sm;
    const int64_t want = (n_rows + rows_per_stage - 1) / rows_per_stage;
    // the narrow kernel is not persistent: one block per row group
    const int64_t blocks = narrow ? (want < int64_t(INT32_MAX) ? want : int64_t(INT32_MAX)) : want < slots ? want : slots;

    BwdParams p{};
    p.dy = static_cast<const char *>(dy);
    p.h = static_cast<const char *>(h);
    p.gamma = static_cast<const char *>(gamma);
    p.dh = static_cast<const char *>(dh);
    p.rstd = rstd;
    p.dx = static_cast<char *>(dx);
    p.dres = static_cast<char *>(dres);
    p.dgamma = dgamma;
    p.sdy = dy_stride * E;
    p.sh = h_stride * E;
    p.sdh = dh_stride * E;
    p.sdx = dx_stride * E;
    p.sdr = dres_stride * E;
    p.rows = n_rows;
    p.H = int(n_cols);
    p.tpr = tpr;
    p.groups = groups;
    p.stages = stages;

    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(unsigned(threads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {&p};
    e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(fn), args);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        cfg.attrs = nullptr;
        cfg.numAttrs = 0;
        e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(fn), args);
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return glu::cuda_fail(e);
    }
    glu_launch_info_t info{};
    info.launched = 1;
    info.backward = 1;
    info.vec_bytes = staged ? 16 : E;
    info.unroll = ept;
    info.threads = threads;
    info.grid = int32_t(blocks);
    info.path = !staged ? 4 : narrow ? 7 : nvt ? 8 : 6;
    info.vector_units = n_rows;
    glu::record_launch(info);
    return GLU_OK;
}
