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
#include "glu_plan.h"

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
