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
// (t + k * threads) * V + i, in a persistent grid (add_rmsnorm_rows_kernel);
// other rows use element accesses at column t + k * threads, one block per row
// (add_rmsnorm_kernel).  Either way consecutive threads touch consecutive
// addresses.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "glu.h"
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
};

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
    int groups;                         // rows a block works on at once
};

__device__ __forceinline__ void red_add_v4(float *p, float a, float b, float c, float d)
{
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

// ds = rstd * gamma * dy - (rstd^3 / H) * s * sum(gamma * dy * s) (+ dh), written
// to dx (and dres); dgamma accumulates dy * s * rstd.  A persistent grid whose
// blocks hold `groups` rows at a time, `tpr` threads per row: each thread owns
// the same columns in every row, so gamma and its dgamma partial sums live in
// registers across the block's rows.  At the end the groups of a block add
// their partial sums in shared memory and the block adds them to dgamma with
// 16-byte reductions, one per 4 columns, so global additions number about
// blocks x H / 4.  The 16-byte path keeps the row's words in registers between
// the row sum and the gradient; the element path reads them again (cache hits),
// which keeps its register count within 1024 threads.  Every element is read
// and written by one thread, reads first, so dx or dres over dy, h or dh is
// safe.
template <class T, int EPT, bool VEC>
__global__ void __launch_bounds__(1024)
    add_rmsnorm_bwd_kernel(const BwdParams p)
{
    using C = Codec<T>;
    constexpr int V = VEC ? 16 / int(sizeof(T)) : 1;
    constexpr int NV = EPT / V;
    constexpr int W = 4;
    extern __shared__ float dsm[];      // [2][groups][33] row sums, then H floats of dgamma (groups > 1)
    const int G = p.groups, tpr = p.tpr;
    float *dgs = dsm + 2 * G * 33;

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const int g = threadIdx.x / tpr, tg = threadIdx.x - g * tpr;
    const int lane = threadIdx.x & 31, wig = tg >> 5, nwg = tpr >> 5;
    const auto column = [&](int k) { return VEC ? (tg + k * tpr) * V : tg + k * tpr; };
    // gamma: the 16-byte path keeps the stored words, the element path fp32 values
    float gam[VEC ? 1 : EPT], dg[EPT];
    uint32_t gw[VEC ? NV : 1][W];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int col = column(k);
#pragma unroll
        for (int i = 0; i < V; ++i) dg[k * V + i] = 0.0f;
        if constexpr (VEC) {
            if (col < p.H) Access<16>::load(p.gamma + int64_t(col) * sizeof(T), gw[k]);
        } else {
            gam[k] = col < p.H ? C::load1(p.gamma + int64_t(col) * sizeof(T)) : 0.0f;
        }
    }
    if (G > 1 && p.dgamma)
        for (int j = threadIdx.x; j < p.H; j += blockDim.x) dgs[j] = 0.0f;

    // the row sum of this thread's group: warp sums, then (one barrier) each
    // thread adds its group's warp sums in order, or for groups of more than 8
    // warps the group's first warp does and a second barrier shares the result
    int parity = 0;
    const auto group_sum = [&](float v) {
        float *r = dsm + (parity * G + g) * 33;
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
    };

    for (int64_t base = int64_t(blockIdx.x) * G; base < p.rows; base += int64_t(gridDim.x) * G, parity ^= 1) {
        const int64_t row = base + g;
        const bool on = row < p.rows;
        const float rs = on ? p.rstd[row] : 0.0f;
        const char *dyr = p.dy + row * p.sdy, *hr = p.h + row * p.sh;
        const char *dhr = p.dh ? p.dh + row * p.sdh : nullptr;
        char *dxr = p.dx + row * p.sdx, *drr = p.dres ? p.dres + row * p.sdr : nullptr;
        SumSq<EPT> dot;
        if constexpr (VEC) {
            uint32_t wd[NV][W], ws[NV][W], we[NV][W];
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int col = column(k);
                if (on && col < p.H) {
                    const int64_t off = int64_t(col) * sizeof(T);
                    Access<16>::load(dyr + off, wd[k]);
                    Access<16>::load(hr + off, ws[k]);
                    if (dhr) Access<16>::load(dhr + off, we[k]);
                }
            }
#pragma unroll
            for (int k = 0; k < NV; ++k)
                if (on && column(k) < p.H)
#pragma unroll
                    for (int j = 0; j < W; ++j)
#pragma unroll
                        for (int e = 0; e < C::kPerWord; ++e) {
                            const int i = k * V + j * C::kPerWord + e;
                            dot.add(i, C::get(gw[k][j], e) * C::get(wd[k][j], e), C::get(ws[k][j], e));
                        }
            const float c = rs * rs * rs * (group_sum(dot.total()) / float(p.H));
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int col = column(k);
                if (on && col < p.H) {
                    uint32_t wo[W];
#pragma unroll
                    for (int j = 0; j < W; ++j) {
                        float f[C::kPerWord];
#pragma unroll
                        for (int e = 0; e < C::kPerWord; ++e) {
                            const int i = k * V + j * C::kPerWord + e;
                            const float d = C::get(wd[k][j], e), sv = C::get(ws[k][j], e);
                            f[e] = rs * C::get(gw[k][j], e) * d - c * sv;
                            if (dhr) f[e] += C::get(we[k][j], e);
                            dg[i] = fmaf(d * sv, rs, dg[i]);
                        }
                        wo[j] = C::put(f);
                    }
                    const int64_t off = int64_t(col) * sizeof(T);
                    Access<16>::store(dxr + off, wo);
                    if (drr) Access<16>::store(drr + off, wo);
                }
            }
        } else {
#pragma unroll
            for (int k = 0; k < EPT; ++k) {
                const int col = column(k);
                if (on && col < p.H) {
                    const int64_t off = int64_t(col) * sizeof(T);
                    dot.add(k, gam[k] * C::load1(dyr + off), C::load1(hr + off));
                }
            }
            const float c = rs * rs * rs * (group_sum(dot.total()) / float(p.H));
#pragma unroll
            for (int k = 0; k < EPT; ++k) {
                const int col = column(k);
                if (on && col < p.H) {
                    const int64_t off = int64_t(col) * sizeof(T);
                    const float d = C::load1(dyr + off), sv = C::load1(hr + off);
                    float v = rs * gam[k] * d - c * sv;
                    if (dhr) v += C::load1(dhr + off);
                    dg[k] = fmaf(d * sv, rs, dg[k]);
                    C::store1(dxr + off, v);
                    if (drr) C::store1(drr + off, v);
                }
            }
        }
    }
    if (!p.dgamma) return;
    const bool v4 = (reinterpret_cast<uintptr_t>(p.dgamma) & 15) == 0;
    if (G == 1) {
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int col = column(k);
            if constexpr (VEC) {
                // V consecutive columns: 16-byte reductions when dgamma allows
#pragma unroll
                for (int i = 0; i < V; i += 4)
                    if (col + i < p.H) {
                        if (v4)
                            red_add_v4(p.dgamma + col + i, dg[k * V + i], dg[k * V + i + 1], dg[k * V + i + 2],
                                       dg[k * V + i + 3]);
                        else
                            for (int q = 0; q < 4; ++q) atomicAdd(p.dgamma + col + i + q, dg[k * V + i + q]);
                    }
            } else {
                if (col < p.H) atomicAdd(p.dgamma + col, dg[k]);
            }
        }
        return;
    }
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int col = column(k);
#pragma unroll
        for (int i = 0; i < V; ++i)
            if (col + i < p.H) atomicAdd(dgs + col + i, dg[k * V + i]);
    }
    __syncthreads();
    for (int j = threadIdx.x * 4; j < p.H; j += blockDim.x * 4) {
        if (v4 && j + 4 <= p.H)
            red_add_v4(p.dgamma + j, dgs[j], dgs[j + 1], dgs[j + 2], dgs[j + 3]);
        else
            for (int q = 0; q < 4 && j + q < p.H; ++q) atomicAdd(p.dgamma + j + q, dgs[j + q]);
    }
}

using BwdFn = void (*)(BwdParams);

BwdFn pick_bwd(int dtype, bool vec)
{
    switch (dtype) {
    case GLU_F32: return vec ? add_rmsnorm_bwd_kernel<float, 8, true> : add_rmsnorm_bwd_kernel<float, 16, false>;
    case GLU_F16: return vec ? add_rmsnorm_bwd_kernel<__half, 16, true> : add_rmsnorm_bwd_kernel<__half, 16, false>;
    default:
        return vec ? add_rmsnorm_bwd_kernel<__nv_bfloat16, 16, true> : add_rmsnorm_bwd_kernel<__nv_bfloat16, 16, false>;
    }
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
    const int E = dtype == GLU_F32 ? 4 : 2;
    if (n_rows == 1) dy_stride = h_stride = dh_stride = dx_stride = dres_stride = n_cols;
    const auto a16 = [](const void *q) { return uintptr_t(q) % 16 == 0; };
    const auto s16 = [E](int64_t st_) { return (st_ * E) % 16 == 0; };
    const int vec_ept = 32 / E;      // 16 elements of 16-bit types, 8 of f32: two 16-byte accesses
    const bool vec = a16(dy) && a16(h) && a16(gamma) && a16(dx) && (!dh || a16(dh)) && (!dres || a16(dres)) &&
                     (n_cols * E) % 16 == 0 && s16(dy_stride) && s16(h_stride) && s16(dx_stride) &&
                     (!dh || s16(dh_stride)) && (!dres || s16(dres_stride)) && n_cols <= int64_t(1024) * vec_ept;
    const int ept = vec ? vec_ept : 16;
    int tpr = int((n_cols + ept - 1) / ept);
    tpr = (tpr + 31) / 32 * 32;
    // narrow rows: several rows per block (up to 512 threads), so that fewer
    // blocks add to dgamma
    const int groups = tpr >= 512 ? 1 : (512 / tpr < 16 ? 512 / tpr : 16);
    const int threads = tpr * groups;
    const size_t smem = sizeof(float) * (size_t(2 * groups * 33) + (groups > 1 ? size_t(n_cols) : 0));
    BwdFn fn = pick_bwd(dtype, vec);

    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reinterpret_cast<const void *>(fn), threads, smem);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return glu::cuda_fail(e);
    }
    const int64_t slots = int64_t(sms) * (per_sm > 0 ? per_sm : 1);
    const int64_t want = (n_rows + groups - 1) / groups;
    const int64_t blocks = want < slots ? want : slots;

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
    info.vec_bytes = vec ? 16 : E;
    info.unroll = ept;
    info.threads = threads;
    info.grid = int32_t(blocks);
    info.path = 4;
    info.vector_units = n_rows;
    glu::record_launch(info);
    return GLU_OK;
}
