// Launch plan shared by the C-ABI front end (glu_api.cu) and the per-dtype
// kernel instantiation units of the streaming kernels.  Host and device see
// the same layout.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace glu {

// One call's work, in bytes and access units.  A "unit" is one full-width
// access per operand (vec_bytes of a, of b, ...); a row of n_cols elements
// holds `vpr` units followed by `rem` tail elements that are handled one at a
// time.  Rows that are contiguous in every operand are walked as one long row.
struct Params {
    const char *a, *b, *dc;       // inputs (dc: backward only)
    char *y0, *y1;                // forward: y0 = y;  backward: y0 = da, y1 = db
    int64_t sa, sb, sdc, sy0, sy1;  // row strides in BYTES
    int64_t rows;
    int64_t vpr;                  // units per row
    int64_t units;                // rows * vpr
    uint32_t div_magic;           // unit -> (row, unit-in-row) by multiply-shift
    uint32_t div_shift;
    int32_t wide;                 // units >= 2^32: plain 64-bit division
    int32_t prefetch;             // ask L2 for the first tile's inputs before waiting on the previous grid
    int64_t rem;                  // tail elements per row (n_cols - vpr * elems-per-unit)
    int64_t tail_units;           // rows * rem
    int64_t tail_col_bytes;       // byte offset of the first tail element in a row
    uint32_t tail_magic;          // tail index -> (row, element-in-tail)
    uint32_t tail_shift;
    int32_t tail_wide;            // tail_units >= 2^32: plain 64-bit division
    int32_t prefetch_ahead;       // > 0: with the prefetch, also the tile this many blocks ahead
};

// Unsigned 32-bit division by a runtime-invariant divisor d >= 1 with one
// high multiply, an add and a shift (Granlund & Montgomery, "Division by
// invariant integers using multiplication", PLDI 1994, section 4): with
// l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
//     n / d == (umulhi(n, m) + n) >> l     for every 32-bit n.
// The sum is formed in 64 bits so it cannot overflow.
inline void fastdiv_init(uint32_t d, uint32_t *magic, uint32_t *shift)
{
    uint32_t l = 0;
    while (l < 32 && (uint64_t(1) << l) < d) ++l;
    uint64_t m = ((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1;
    *magic = uint32_t(m);   // m < 2^32 for every d >= 1
    *shift = l;
}

__host__ __device__ inline uint32_t fastdiv(uint32_t n, uint32_t magic, uint32_t shift)
{
#ifdef __CUDA_ARCH__
    uint32_t hi = __umulhi(n, magic);
#else
    uint32_t hi = uint32_t((uint64_t(n) * magic) >> 32);
#endif
    return uint32_t((uint64_t(hi) + n) >> shift);
}

enum Dir { kFwd = 0, kBwd = 1 };

using KernelFn = void (*)(Params);

// Per-dtype kernel tables, defined in the instantiation units.  `vb_sel`:
// 0 = 32-byte units, 1 = 16-byte units, 2 = one element per unit;
// `unroll_sel`: 0, 1, 2 for 1, 2, 4 units in flight per operand per thread.
KernelFn kernel_f32(int act, int dir, int vb_sel, int unroll_sel);
KernelFn kernel_f16(int act, int dir, int vb_sel, int unroll_sel);
KernelFn kernel_bf16(int act, int dir, int vb_sel, int unroll_sel);

constexpr int kThreads = 256;

}  // namespace glu
