// Streaming kernels of the gated activation: one template per direction,
// instantiated per (activation, dtype, access width, accesses in flight).
//
// Decomposition ("Skill: Write a Triton SiLU-Mul (SwiGLU) Kernel", Required
// reasoning process steps 1-3, and "Kernel Profile: SwiGLU", Tiling Strategy,
// redone for sm_103a): the work is a flat index space of `units`, each unit a
// 32- or 16-byte access per operand inside one row.  A block takes a tile of
// kThreads * UNROLL consecutive units (consecutive threads -> consecutive
// units, so every warp access is coalesced), issues all of its loads before
// any arithmetic (UNROLL * operands accesses in flight per thread), converts to
// fp32, applies the activation, rounds once to the storage dtype and stores.
// Unit -> (row, byte offset) is one multiply-shift division per unit; rows that
// are contiguous in every operand are walked as one row.  The elements at the
// end of a row that do not fill a unit ("mask every load and the store",
// step 2) form a separate scalar tail.
//
// In place: every element's loads precede its stores in the same thread and
// units never overlap, so an output may be the same matrix as an input
// ("Common failure modes", in-place store before the load completes;
// "Kernel Profile: SwiGLU", Key Patterns, in-place backward).  The accesses are
// volatile inline PTX with a memory clobber, so the compiler keeps that order.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "glu_math.cuh"
#include "glu_plan.h"

namespace glu {

// ---------------------------------------------------------------- memory access
// L1::no_allocate: every byte is touched once, so nothing is kept in L1.

template <int VB>
struct Access;

template <>
struct Access<16> {
    static constexpr int W = 4;
    __device__ __forceinline__ static void load(const char *p, uint32_t (&w)[4])
    {
        asm volatile("ld.global.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                     : "l"(p)
                     : "memory");
    }
    __device__ __forceinline__ static void store(char *p, const uint32_t (&w)[4])
    {
        asm volatile("st.global.L1::no_allocate.v4.b32 [%0], {%1,%2,%3,%4};"
                     :
                     : "l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                     : "memory");
    }
};

template <>
struct Access<32> {   // 256-bit global accesses (sm_100 and later)
    static constexpr int W = 8;
    __device__ __forceinline__ static void load(const char *p, uint32_t (&w)[8])
    {
        asm volatile("ld.global.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]),
                       "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                     : "l"(p)
                     : "memory");
    }
    __device__ __forceinline__ static void store(char *p, const uint32_t (&w)[8])
    {
        asm volatile("st.global.L1::no_allocate.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                     :
                     : "l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]),
                       "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                     : "memory");
    }
};

// ---------------------------------------------------------------- dtype codecs
// Storage <-> fp32.  Narrowing is round-to-nearest-even with IEEE overflow to
// infinity and gradual underflow ("cast back to the storage dtype only at the
// final store").

template <class T>
struct Codec;

template <>
struct Codec<float> {
    static constexpr int kPerWord = 1;
    __device__ __forceinline__ static float get(uint32_t w, int) { return __uint_as_float(w); }
    __device__ __forceinline__ static uint32_t put(const float *f) { return __float_as_uint(f[0]); }
    __device__ __forceinline__ static float load1(const char *p)
    {
        uint32_t v;
        asm volatile("ld.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
        return __uint_as_float(v);
    }
    __device__ __forceinline__ static void store1(char *p, float f)
    {
        asm volatile("st.global.b32 [%0], %1;" ::"l"(p), "r"(__float_as_uint(f)) : "memory");
    }
};

template <>
struct Codec<__nv_bfloat16> {
    static constexpr int kPerWord = 2;
    __device__ __forceinline__ static float get(uint32_t w, int j)
    {
        return __uint_as_float(j ? (w & 0xFFFF0000u) : (w << 16));
    }
    __device__ __forceinline__ static uint32_t put(const float *f)
    {
        __nv_bfloat162 h = __floats2bfloat162_rn(f[0], f[1]);   // .x (low half) = f[0]
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ __forceinline__ static float load1(const char *p)
    {
        unsigned short v;
        asm volatile("ld.global.b16 %0, [%1];" : "=h"(v) : "l"(p) : "memory");
        return __uint_as_float(uint32_t(v) << 16);
    }
    __device__ __forceinline__ static void store1(char *p, float f)
    {
        unsigned short v = __bfloat16_as_ushort(__float2bfloat16_rn(f));
        asm volatile("st.global.b16 [%0], %1;" ::"l"(p), "h"(v) : "memory");
    }
};

template <>
struct Codec<__half> {
    static constexpr int kPerWord = 2;
    __device__ __forceinline__ static float get(uint32_t w, int j)
    {
        return __half2float(__ushort_as_half((unsigned short)(j ? (w >> 16) : (w & 0xFFFFu))));
    }
    __device__ __forceinline__ static uint32_t put(const float *f)
    {
        __half2 h = __floats2half2_rn(f[0], f[1]);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ __forceinline__ static float load1(const char *p)
    {
        unsigned short v;
        asm volatile("ld.global.b16 %0, [%1];" : "=h"(v) : "l"(p) : "memory");
        return __half2float(__ushort_as_half(v));
    }
    __device__ __forceinline__ static void store1(char *p, float f)
    {
        unsigned short v = __half_as_ushort(__float2half_rn(f));
        asm volatile("st.global.b16 [%0], %1;" ::"l"(p), "h"(v) : "memory");
    }
};

// ---------------------------------------------------------------- index maps

// unit u -> (row, byte offset of the unit inside the row)
template <int VB>
__device__ __forceinline__ void unit_pos(const Params &p, int64_t u, int64_t &row, int64_t &cb)
{
    if (p.rows == 1) {
        row = 0;
        cb = u * VB;
    } else if (!p.wide) {
        uint32_t q = fastdiv(uint32_t(u), p.div_magic, p.div_shift);
        row = q;
        cb = int64_t(uint32_t(u) - q * uint32_t(p.vpr)) * VB;
    } else {
        row = u / p.vpr;
        cb = (u - row * p.vpr) * VB;
    }
}

// ---------------------------------------------------------------- element ops

template <class Act, bool Exact>
__device__ __forceinline__ float op_fwd(float a, float b)
{
    return Act::template fwd<Exact>(a) * b;                    // y = act(a) * b
}

template <class Act, bool Exact>
__device__ __forceinline__ void op_bwd(float c, float a, float b, float &da, float &db)
{
    float s, ds;
    Act::template bwd<Exact>(a, &s, &ds);
    da = c * ds * b;                                           // dc * act'(a) * b
    db = c * s;                                                // dc * act(a)
}

// One storage word of the forward (1 or 2 elements): y = act(a) * b; a
// 16-bit word's two elements as one pair.
template <class Act, bool Exact, class Cd, int PW = Cd::kPerWord>
__device__ __forceinline__ void fwd_word(uint32_t wa, uint32_t wb, float (&y)[PW])
{
    if constexpr (PW == 2) {
        const f2 a = make_float2(Cd::get(wa, 0), Cd::get(wa, 1));
        const f2 b = make_float2(Cd::get(wb, 0), Cd::get(wb, 1));
        const f2 r = mul2(Act::fwd2(a), b);                    // act(a) * b
        y[0] = r.x;
        y[1] = r.y;
    } else {
        y[0] = op_fwd<Act, Exact>(Cd::get(wa, 0), Cd::get(wb, 0));
    }
}

// One storage word of the backward (1 or 2 elements): act and act' for every
// element, the root series only on the rare path where an element lies next
// to a root of act', then da = dc act' b and db = dc act.
template <class Act, bool Exact, class Cd, int PW = Cd::kPerWord>
__device__ __forceinline__ void bwd_word(uint32_t wa, uint32_t wb, uint32_t wc, float (&da)[PW],
                                         float (&db)[PW])
{
    if constexpr (PW == 2) {
        const f2 a = make_float2(Cd::get(wa, 0), Cd::get(wa, 1));
        f2 s, ds;
        Act::bwd2(a, &s, &ds);
        if (Act::near_root(a.x) || Act::near_root(a.y)) {
            Act::fix_root(a.x, &ds.x);
            Act::fix_root(a.y, &ds.y);
        }
        const f2 c = make_float2(Cd::get(wc, 0), Cd::get(wc, 1));
        const f2 b = make_float2(Cd::get(wb, 0), Cd::get(wb, 1));
        const f2 ra = mul2(mul2(c, ds), b);                    // dc * act'(a) * b
        const f2 rb = mul2(c, s);                              // dc * act(a)
        da[0] = ra.x;
        da[1] = ra.y;
        db[0] = rb.x;
        db[1] = rb.y;
    } else {
        float s, ds;
        const float a = Cd::get(wa, 0);
        Act::template bwd_main<Exact>(a, &s, &ds);
        if (Act::near_root(a)) Act::fix_root(a, &ds);
        const float c = Cd::get(wc, 0), b = Cd::get(wb, 0);
        da[0] = c * ds * b;                                    // dc * act'(a) * b
        db[0] = c * s;                                         // dc * act(a)
    }
}

// ---------------------------------------------------------------- L2 prefetch
// One prefetch per 128-byte line of this block's first tile of inputs (the
// lane whose unit holds the line's start), and with p.prefetch_ahead = the
// blocks resident at once, of the tile one wave ahead too, which a block of
// the second wave would otherwise only ask for once it starts.  L2 is the
// device's point of coherence, so a line the previous grid writes after the
// prefetch is updated there, and loads issued after griddepcontrol.wait still
// see its data: the prefetch only lets DRAM start on this launch's inputs
// during the previous launch's last wave.  Not inlined, so that its address
// arithmetic does not stay live into the kernel's main loop (inlined, it cost
// the forward kernel a block per SM).
template <int VB, int UNROLL, int DIR>
__device__ __noinline__ void prefetch_first_tile(const Params &p)
{
    const int n = p.prefetch_ahead > 0 ? 2 * UNROLL : UNROLL;
    for (int k = 0; k < n; ++k) {
        const int64_t tb = int64_t(blockIdx.x) + (k >= UNROLL ? int64_t(p.prefetch_ahead) : 0);
        const int64_t u = tb * kThreads * UNROLL + (k % UNROLL) * kThreads + threadIdx.x;
        if (u >= p.units) continue;
        int64_t row, cb;
        unit_pos<VB>(p, u, row, cb);
        const char *pa = p.a + row * p.sa + cb, *pb = p.b + row * p.sb + cb;
        if ((reinterpret_cast<uintptr_t>(pa) & 127) < VB) asm volatile("prefetch.global.L2 [%0];" ::"l"(pa));
        if ((reinterpret_cast<uintptr_t>(pb) & 127) < VB) asm volatile("prefetch.global.L2 [%0];" ::"l"(pb));
        if constexpr (DIR == kBwd) {
            const char *pc = p.dc + row * p.sdc + cb;
            if ((reinterpret_cast<uintptr_t>(pc) & 127) < VB) asm volatile("prefetch.global.L2 [%0];" ::"l"(pc));
        }
    }
}

// ---------------------------------------------------------------- the kernel
// DIR = kFwd: (a, b) -> y0.   DIR = kBwd: (dc, a, b) -> (y0 = da, y1 = db).
// VB = 32 or 16: vector units then the scalar tail; VB = 0: scalar tail only.

template <class Act, class T, int VB, int UNROLL, int DIR>
__global__ void __launch_bounds__(kThreads) glu_kernel(const Params p)
{
    constexpr bool kExact = std::is_same<T, float>::value;
    using C = Codec<T>;

    // Programmatic dependent launch: let the next kernel in the stream be
    // scheduled while this grid's last blocks run, and do not touch memory
    // before the previous grid has completed and its writes are visible.
    // Both are no-ops when the launch carries no programmatic dependency.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // Small launches (p.prefetch): before waiting for the previous grid, ask
    // L2 for this block's first tile of inputs (prefetch_first_tile).  Large
    // launches keep DRAM busy through the previous launch's last wave anyway
    // and measured slower with it.
    if (VB > 0 && p.prefetch) prefetch_first_tile<VB, UNROLL, DIR>(p);
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if constexpr (VB > 0) {
        constexpr int W = Access<VB>::W;
        constexpr int PW = C::kPerWord;
        constexpr int64_t kTile = int64_t(kThreads) * UNROLL;
        const int64_t step = int64_t(gridDim.x) * kTile;
        for (int64_t t0 = int64_t(blockIdx.x) * kTile; t0 < p.units; t0 += step) {
            uint32_t va[UNROLL][W], vb[UNROLL][W], vc[UNROLL][DIR == kBwd ? W : 1];
            int64_t rows[UNROLL], cbs[UNROLL];
#pragma unroll
            for (int k = 0; k < UNROLL; ++k) {
                const int64_t u = t0 + k * kThreads + threadIdx.x;
                if (u < p.units) {
                    unit_pos<VB>(p, u, rows[k], cbs[k]);
                    if constexpr (DIR == kBwd) Access<VB>::load(p.dc + rows[k] * p.sdc + cbs[k], vc[k]);
                    Access<VB>::load(p.a + rows[k] * p.sa + cbs[k], va[k]);
                    Access<VB>::load(p.b + rows[k] * p.sb + cbs[k], vb[k]);
                }
            }
#pragma unroll
            for (int k = 0; k < UNROLL; ++k) {
                const int64_t u = t0 + k * kThreads + threadIdx.x;
                if (u < p.units) {
                    uint32_t o0[W], o1[DIR == kBwd ? W : 1];
#pragma unroll
                    for (int j = 0; j < W; ++j) {
                        float f0[PW], f1[PW];
                        if constexpr (DIR == kFwd) {
                            fwd_word<Act, kExact, C>(va[k][j], vb[k][j], f0);
                        } else {
                            bwd_word<Act, kExact, C>(va[k][j], vb[k][j], vc[k][j], f0, f1);
                        }
                        o0[j] = C::put(f0);
                        if constexpr (DIR == kBwd) o1[j] = C::put(f1);
                    }
                    Access<VB>::store(p.y0 + rows[k] * p.sy0 + cbs[k], o0);
                    if constexpr (DIR == kBwd) Access<VB>::store(p.y1 + rows[k] * p.sy1 + cbs[k], o1);
                }
            }
        }
    }

    // Scalar tail: the last `rem` elements of every row (all elements when VB == 0).
    const int64_t tstep = int64_t(gridDim.x) * kThreads;
    for (int64_t t = int64_t(blockIdx.x) * kThreads + threadIdx.x; t < p.tail_units; t += tstep) {
        int64_t row, j;
        if (p.rows == 1) {
            row = 0;
            j = t;
        } else if (!p.tail_wide) {
            uint32_t q = fastdiv(uint32_t(t), p.tail_magic, p.tail_shift);
            row = q;
            j = int64_t(uint32_t(t) - q * uint32_t(p.rem));
        } else {
            row = t / p.rem;
            j = t - row * p.rem;
        }
        const int64_t cb = p.tail_col_bytes + j * int64_t(sizeof(T));
        const float a = C::load1(p.a + row * p.sa + cb);
        const float b = C::load1(p.b + row * p.sb + cb);
        if constexpr (DIR == kFwd) {
            C::store1(p.y0 + row * p.sy0 + cb, op_fwd<Act, kExact>(a, b));
        } else {
            const float c = C::load1(p.dc + row * p.sdc + cb);
            float da, db;
            op_bwd<Act, kExact>(c, a, b, da, db);
            C::store1(p.y0 + row * p.sy0 + cb, da);
            C::store1(p.y1 + row * p.sy1 + cb, db);
        }
    }
}

// ---------------------------------------------------------------- tables

template <class T, class Act, int DIR>
KernelFn pick(int vb_sel, int unroll_sel)
{
    switch (vb_sel * 3 + unroll_sel) {
    case 0: return glu_kernel<Act, T, 32, 1, DIR>;
    case 1: return glu_kernel<Act, T, 32, 2, DIR>;
    case 2: return glu_kernel<Act, T, 32, 4, DIR>;
    case 3: return glu_kernel<Act, T, 16, 1, DIR>;
    case 4: return glu_kernel<Act, T, 16, 2, DIR>;
    case 5: return glu_kernel<Act, T, 16, 4, DIR>;
    default: return glu_kernel<Act, T, 0, 1, DIR>;
    }
}

template <class T, class Act>
KernelFn pick_dir(int dir, int vb_sel, int unroll_sel)
{
    return dir == kBwd ? pick<T, Act, kBwd>(vb_sel, unroll_sel) : pick<T, Act, kFwd>(vb_sel, unroll_sel);
}

template <class T>
KernelFn select_kernel(int act, int dir, int vb_sel, int unroll_sel)
{
    switch (act) {
    case 0: return pick_dir<T, Silu>(dir, vb_sel, unroll_sel);
    case 1: return pick_dir<T, GeluErf>(dir, vb_sel, unroll_sel);
    case 2: return pick_dir<T, GeluTanh>(dir, vb_sel, unroll_sel);
    case 3: return pick_dir<T, Relu>(dir, vb_sel, unroll_sel);
    default: return nullptr;
    }
}

}  // namespace glu
