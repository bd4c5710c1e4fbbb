// C-ABI front end: argument validation, aliasing rules, launch planning and
// dispatch to the per-dtype kernel tables.  Declarations and the contract of
// every entry point are in include/glu.h.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstring>

#include "glu.h"
#include "glu_async.cuh"
#include "glu_internal.h"

namespace {

using glu::kBwd;
using glu::kFwd;
using glu::Params;

thread_local glu_launch_info_t t_last_launch{};
thread_local char t_cuda_error[256] = "";

// Process-wide tuning; 0 = library default.
std::atomic<int32_t> g_vec_bytes{0};
std::atomic<int32_t> g_unroll{0};
std::atomic<int32_t> g_ctas_per_sm{0};
std::atomic<int32_t> g_dependent_launch{0};
std::atomic<int32_t> g_path{0};                // 0 default, 1 direct loads, 2 bulk copies
constexpr int32_t kDefaultCtasPerSm = -1;     // one block per tile

// Default access width (bytes) and accesses in flight per operand per thread,
// by [dtype][activation][direction], from a sweep on GB300 of 4096 x {4096,
// 16384} matrices launched back to back: the forward of the heavier GELUs wants
// two 32-byte accesses in flight (more arithmetic to hide), the 16-bit SiLU,
// GeGLU-erf and GeGLU-tanh backward two 16-byte ones, ReGLU one 32-byte access
// (5-12 % ahead of one 16-byte access on its forward at every width and dtype in
// alternating runs, level or ahead on its backward).  Re-swept at 4096 x {1024
// ... 16384}: the 16-bit GeGLU-erf backward 7-9 % faster with two 16-byte
// accesses than with one 32-byte access at every width; the f32 SiLU backward
// 5 % faster at 1024 with one 32-byte access, level (within 0.6 %) above.
struct LaunchDefault {
    int8_t vec_bytes, unroll;
};
constexpr LaunchDefault kDefaults[3][4][2] = {
    // f32:  silu            gelu_erf         gelu_tanh        relu
    {{{32, 1}, {32, 1}}, {{32, 2}, {32, 1}}, {{32, 2}, {32, 1}}, {{32, 1}, {32, 1}}},
    // f16
    {{{32, 1}, {16, 2}}, {{32, 2}, {16, 2}}, {{32, 2}, {16, 2}}, {{32, 1}, {32, 1}}},
    // bf16
    {{{32, 1}, {16, 2}}, {{32, 2}, {16, 2}}, {{32, 2}, {16, 2}}, {{32, 1}, {32, 1}}},
};

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

int elem_size(int dtype) { return dtype == GLU_F32 ? 4 : 2; }

bool valid_enums(int layout, int act, int dtype)
{
    return (layout == GLU_LAYOUT_SPLIT || layout == GLU_LAYOUT_CONCAT) &&
           (act >= GLU_ACT_SILU && act <= GLU_ACT_RELU) &&
           (dtype == GLU_F32 || dtype == GLU_F16 || dtype == GLU_BF16);
}

// A matrix operand: base address, row stride and row width in elements.
struct Mat {
    uintptr_t p;
    int64_t stride;
    int64_t width;
};

// Byte extent of a matrix: ((rows - 1) * stride + width) * E, or -1 on overflow.
int64_t extent_bytes(const Mat &m, int64_t rows, int E)
{
    int64_t last, span, bytes;
    if (__builtin_mul_overflow(rows - 1, m.stride, &last)) return -1;
    if (__builtin_add_overflow(last, m.width, &span)) return -1;
    if (__builtin_mul_overflow(span, int64_t(E), &bytes)) return -1;
    if (uint64_t(bytes) > UINTPTR_MAX - m.p) return -1;
    return bytes;
}

// Do the element sets of X and Y (same rows, same width C, element size E)
// share an address?  Exact for equal strides; conservative (overlapping
// footprints count as overlap) otherwise.
bool elems_overlap(const Mat &X, const Mat &Y, int64_t rows, int E)
{
    const uint64_t x0 = X.p, x1 = X.p + uint64_t(extent_bytes(X, rows, E));
    const uint64_t y0 = Y.p, y1 = Y.p + uint64_t(extent_bytes(Y, rows, E));
    if (x1 <= y0 || y1 <= x0) return false;
    if (rows == 1 || X.stride != Y.stride) return true;
    const int64_t diff = int64_t(Y.p - X.p);
    if (diff % E != 0) return true;
    // Y's (r, c) is X's element d + r*s + c.  A shared element needs a row
    // offset k with |k| < rows and |d - k s| < C; since C <= s only
    // k = floor(d / s) and k + 1 can qualify.
    const int64_t d = diff / E, s = X.stride, C = X.width;
    int64_t k = d / s;
    if ((d % s != 0) && ((d < 0) != (s < 0))) --k;          // floor division
    for (int64_t kk = k; kk <= k + 1; ++kk) {
        const int64_t r = d - kk * s;
        if ((kk < rows && -kk < rows) && (r < C && -r < C)) return true;
    }
    return false;
}

// Does any of the rows of M (each width * E bytes) share a byte with [p, p + len)?
bool rows_hit_range(const Mat &M, int64_t rows, int E, uint64_t p, uint64_t len)
{
    const uint64_t m0 = M.p, m1 = M.p + uint64_t(extent_bytes(M, rows, E));
    if (m1 <= p || p + len <= m0) return false;
    if (rows == 1) return true;
    const uint64_t pitch = uint64_t(M.stride) * E, w = uint64_t(M.width) * E;
    const uint64_t first = p > m0 ? (p - m0) / pitch : 0;      // the row at or before p
    for (uint64_t r = first; r < uint64_t(rows) && m0 + r * pitch < p + len; ++r)
        if (m0 + r * pitch + w > p) return true;
    return false;
}

bool same_mat(const Mat &X, const Mat &Y, int64_t rows)
{
    return X.p == Y.p && (rows == 1 || X.stride == Y.stride) && X.width == Y.width;
}

// Outputs may equal an input exactly; any other overlap is an error, and two
// outputs may not overlap at all.
int check_aliasing(const Mat *in, int n_in, const Mat *out, int n_out, int64_t rows, int E)
{
    for (int o = 0; o < n_out; ++o) {
        for (int i = 0; i < n_in; ++i)
            if (!same_mat(out[o], in[i], rows) && elems_overlap(out[o], in[i], rows, E))
                return GLU_ERR_ALIAS;
        for (int q = o + 1; q < n_out; ++q)
            if (elems_overlap(out[o], out[q], rows, E)) return GLU_ERR_ALIAS;
    }
    return GLU_OK;
}

int sm_count()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
    if (dev < kMaxDevices) {
        int c = g_sm_count[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int c = 0;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    if (dev < kMaxDevices) g_sm_count[dev].store(c, std::memory_order_relaxed);
    return c;
}

// Blocks of glu::kThreads threads of kernel `fn` resident on one SM at once,
// asked once per device and kernel variant (`key` < 216: dtype, activation,
// direction, access width, accesses in flight); 0 if the query fails.
// Devices numbered 64 and above are asked on every call.
std::atomic<int> g_resident[kMaxDevices][216];

int resident_blocks(const void *fn, int key)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    if (dev >= 0 && dev < kMaxDevices) {
        const int c = g_resident[dev][key].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int per = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, fn, glu::kThreads, 0) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    if (dev >= 0 && dev < kMaxDevices && per > 0) g_resident[dev][key].store(per, std::memory_order_relaxed);
    return per;
}

using glu::cuda_fail;

using glu::Call;

// Launches `fn` with the programmatic-dependency attribute unless switched
// off; falls back to an ordinary launch if the runtime refuses the attribute.
cudaError_t launch_kernel(const void *fn, dim3 grid, dim3 block, size_t smem, void **args,
                          cudaStream_t stream)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    const bool dependent = g_dependent_launch.load(std::memory_order_relaxed) >= 0;
    cfg.attrs = dependent ? attr : nullptr;
    cfg.numAttrs = dependent ? 1 : 0;
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess && dependent) {
        (void)cudaGetLastError();
        cfg.attrs = nullptr;
        cfg.numAttrs = 0;
        e = cudaLaunchKernelExC(&cfg, fn, args);
    }
    return e;
}

int plan_direct(const Call &c, cudaStream_t stream);

// Bulk-copy staging path: contiguous operands, 16-byte aligned, inputs in
// device memory, at least one whole chunk.  Whole chunks go to the bulk kernel
// (one block per SM), the remainder to the direct kernel.  Returns 1 if the
// call is not eligible.
int plan_bulk(const Call &c, cudaStream_t stream)
{
    const int n_ops = c.dir == kBwd ? 5 : 3;
    const uintptr_t ptrs[5] = {uintptr_t(c.a), uintptr_t(c.b), uintptr_t(c.y0), uintptr_t(c.dc),
                               uintptr_t(c.y1)};
    const int64_t strides[5] = {c.sa, c.sb, c.sy0, c.sdc, c.sy1};
    bool flat = true;
    for (int i = 0; i < n_ops; ++i) {
        flat = flat && (c.rows == 1 || strides[i] == c.cols);
        flat = flat && (ptrs[i] % 16 == 0);
    }
    const int64_t bytes = c.rows * c.cols * c.E;
    const int64_t chunks = bytes / glu::kBulkChunkHost;
    if (!flat || chunks < 1) return 1;
    // the bulk-copy engine is given device memory only: inputs anywhere else
    // (pinned host memory included) take the direct path
    const void *inputs[3] = {c.a, c.b, c.dir == kBwd ? c.dc : nullptr};
    for (const void *q : inputs) {
        if (!q) continue;
        bool dev_mem = false;
        const cudaError_t pe = glu::on_device(q, &dev_mem);
        if (pe != cudaSuccess) return glu::cuda_fail(pe);
        if (!dev_mem) return 1;
    }

    // ctas_per_sm 1 selects the wide shape, anything else the narrow one
    const bool narrow = g_ctas_per_sm.load(std::memory_order_relaxed) != 1;
    static std::atomic<int> smem_set[3][4][2][2];
    glu::BulkFn fn = glu::bulk_kernel(c.dtype, c.act, c.dir, narrow);
    if (!fn) return GLU_ERR_ENUM;
    const int smem = glu::bulk_smem_bytes(c.dir, narrow);
    std::atomic<int> &flag = smem_set[c.dtype][c.act][c.dir][narrow];
    if (!flag.load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void *>(fn),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) { (void)cudaGetLastError(); return cuda_fail(e); }
        flag.store(1, std::memory_order_release);
    }
    const int sms = sm_count();
    if (sms <= 0) return cuda_fail(cudaGetLastError());
    glu::BulkParams bp{c.a, c.b, c.dc, c.y0, c.y1, chunks};
    void *args[] = {&bp};
    const int64_t slots = int64_t(sms) * (narrow ? 2 : 1);
    const int64_t grid = chunks < slots ? chunks : slots;
    const int threads = glu::bulk_threads(narrow);
    cudaError_t e = launch_kernel(reinterpret_cast<const void *>(fn), dim3(unsigned(grid)),
                                  dim3(threads), size_t(smem), args, stream);
    if (e != cudaSuccess) { (void)cudaGetLastError(); return cuda_fail(e); }

    glu_launch_info_t info{};
    info.launched = 1;
    info.backward = c.dir == kBwd;
    info.vec_bytes = 16;
    info.unroll = 1;
    info.threads = threads;
    info.grid = int32_t(grid);
    info.flattened = c.rows > 1;
    info.path = 2;
    info.vector_units = chunks * (glu::kBulkChunkHost / 16);
    const int64_t done_elems = chunks * glu::kBulkChunkHost / c.E;
    const int64_t rest = c.rows * c.cols - done_elems;
    info.tail_elems = rest;
    if (rest > 0) {
        Call r = c;
        const int64_t off = done_elems * c.E;
        r.rows = 1;
        r.cols = rest;
        r.a = c.a + off; r.b = c.b + off; r.y0 = c.y0 + off;
        if (c.dir == kBwd) { r.dc = c.dc + off; r.y1 = c.y1 + off; }
        r.sa = r.sb = r.sy0 = r.sdc = r.sy1 = rest;
        const int st = plan_direct(r, stream);
        if (st != GLU_OK) return st;
    }
    t_last_launch = info;
    return GLU_OK;
}

int plan_and_launch(const Call &c, cudaStream_t stream)
{
    if (g_path.load(std::memory_order_relaxed) == 2) {
        const int st = plan_bulk(c, stream);
        if (st != 1) return st;
    }
    return plan_direct(c, stream);
}

int plan_direct(const Call &c, cudaStream_t stream)
{
    const int E = c.E;
    const int n_ops = c.dir == glu::kBwd ? 5 : 3;
    const uintptr_t ptrs[5] = {uintptr_t(c.a), uintptr_t(c.b), uintptr_t(c.y0),
                               uintptr_t(c.dc), uintptr_t(c.y1)};
    const int64_t strides[5] = {c.sa, c.sb, c.sy0, c.sdc, c.sy1};

    // Rows that are contiguous in every operand are one long row.
    bool flat = c.rows == 1;
    if (!flat) {
        flat = true;
        for (int i = 0; i < n_ops; ++i) flat = flat && strides[i] == c.cols;
    }
    const int64_t R = flat ? 1 : c.rows;
    const int64_t C = flat ? c.rows * c.cols : c.cols;   // fits: extents were checked

    // Widest access every operand's rows are aligned to.
    int32_t cap = g_vec_bytes.load(std::memory_order_relaxed);
    const LaunchDefault dflt = kDefaults[c.dtype][c.act][c.dir];
    if (cap == 0) cap = dflt.vec_bytes;
    int vb = 0;
    for (int cand : {32, 16}) {
        if (cand > cap) continue;
        bool ok = true;
        for (int i = 0; i < n_ops; ++i) {
            ok = ok && (ptrs[i] % cand == 0);
            if (!flat) ok = ok && ((strides[i] * E) % cand == 0);
        }
        if (ok) { vb = cand; break; }
    }
    int32_t unroll = g_unroll.load(std::memory_order_relaxed);
    if (unroll == 0) {
        // Matrices of up to 2^22 elements fill only one or two waves of
        // blocks; one access in flight per thread doubles the blocks and
        // evens out the last wave.
        unroll = c.rows * c.cols <= (int64_t(1) << 22) ? 1 : dflt.unroll;
    }
    const int unroll_sel = unroll == 1 ? 0 : (unroll == 2 ? 1 : 2);
    const int vb_sel = vb == 32 ? 0 : (vb == 16 ? 1 : 2);
    if (vb == 0) unroll = 1;

    Params p{};
    p.a = c.a; p.b = c.b; p.dc = c.dc; p.y0 = c.y0; p.y1 = c.y1;
    p.sa = c.sa * E; p.sb = c.sb * E; p.sdc = c.sdc * E; p.sy0 = c.sy0 * E; p.sy1 = c.sy1 * E;
    p.rows = R;
    const int64_t per_unit = vb ? vb / E : 0;
    p.vpr = per_unit ? C / per_unit : 0;
    p.units = R * p.vpr;
    p.rem = C - p.vpr * per_unit;
    p.tail_units = R * p.rem;
    p.tail_col_bytes = p.vpr * vb;
    p.wide = p.units >= (int64_t(1) << 32);
    if (p.units > 0 && R > 1 && !p.wide) glu::fastdiv_init(uint32_t(p.vpr), &p.div_magic, &p.div_shift);
    p.tail_wide = p.tail_units >= (int64_t(1) << 32);
    // Inputs of at most 64 MiB: the L2 prefetch before the dependency wait
    // (glu_kernels.cuh).  Measured back to back on GB300 against the same
    // build without it (interleaved): bf16 SwiGLU forward +4.6 % at
    // 4096 x 1024, +5.2 % at 4096 x 2048, +2.4 % at 4096 x 4096; backward
    // +4.3 % at 4096 x 1024; GeGLU-erf and f32 forwards at 4096 x 1024 +4-5 %;
    // the backward at 4096 x 4096 (96 MiB of inputs) -0.8 %, and larger
    // launches, whose predecessor's last wave keeps DRAM busy anyway, -1 to
    // -2 % when it was on for them.
    p.prefetch = int64_t(c.dir == glu::kBwd ? 3 : 2) * c.rows * c.cols * E <= (int64_t(64) << 20);
    if (p.tail_units > 0 && R > 1 && !p.tail_wide) glu::fastdiv_init(uint32_t(p.rem), &p.tail_magic, &p.tail_shift);

    glu::KernelFn fn = nullptr;
    switch (c.dtype) {
    case GLU_F32: fn = glu::kernel_f32(c.act, c.dir, vb_sel, unroll_sel); break;
    case GLU_F16: fn = glu::kernel_f16(c.act, c.dir, vb_sel, unroll_sel); break;
    default: fn = glu::kernel_bf16(c.act, c.dir, vb_sel, unroll_sel); break;
    }
    if (!fn) return GLU_ERR_ENUM;

    // Grid: one block per tile of kThreads * unroll units (and enough blocks
    // for the scalar tail), or a persistent grid of ctas_per_sm blocks per SM.
    const int64_t tile = int64_t(glu::kThreads) * unroll;
    int64_t blocks = (p.units + tile - 1) / tile;
    const int64_t tail_blocks = (p.tail_units + glu::kThreads - 1) / glu::kThreads;
    if (tail_blocks > blocks) blocks = tail_blocks;
    if (blocks < 1) blocks = 1;
    int32_t per_sm = g_ctas_per_sm.load(std::memory_order_relaxed);
    if (per_sm == 0) per_sm = kDefaultCtasPerSm;
    if (per_sm > 0) {
        const int sms = sm_count();
        if (sms <= 0) return cuda_fail(cudaGetLastError());
        if (blocks > int64_t(per_sm) * sms) blocks = int64_t(per_sm) * sms;
    }
    if (blocks > 0x7FFFFFFF) blocks = 0x7FFFFFFF;
    // Forward launches of at most 16 MiB of inputs and more blocks than SMs:
    // the blocks of the first wave also prefetch the tile one wave ahead
    // (glu_kernels.cuh).  Measured back to back against the same build without
    // it (interleaved): 4096 x 1024 bf16 SiLU / GeGLU-erf / ReGLU forward and
    // 2048 x 2048 SiLU 3-5 % faster; on the backward and on 32-48 MiB
    // forwards it was up to 7 % slower.
    if (p.prefetch && c.dir == glu::kFwd && int64_t(2) * c.rows * c.cols * E <= (int64_t(16) << 20)) {
        const int sms = sm_count();
        if (sms > 0 && blocks > sms) {
            const int key = (((c.dtype * 4 + c.act) * 2 + c.dir) * 3 + vb_sel) * 3 + unroll_sel;
            const int per = resident_blocks(reinterpret_cast<const void *>(fn), key);
            if (per > 0) p.prefetch_ahead = per * sms;
        }
    }

    // Launch with a programmatic dependency on the previous kernel in the
    // stream (unless switched off): the kernel waits for that grid itself, so
    // ordering and visibility are unchanged, but its blocks can be scheduled
    // during the previous grid's tail.
    void *args[] = {&p};
    cudaError_t e = launch_kernel(reinterpret_cast<const void *>(fn), dim3(unsigned(blocks)),
                                  dim3(glu::kThreads), 0, args, stream);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return cuda_fail(e);
    }

    glu_launch_info_t info{};
    info.launched = 1;
    info.backward = c.dir == glu::kBwd;
    info.vec_bytes = vb ? vb : E;
    info.unroll = unroll;
    info.threads = glu::kThreads;
    info.grid = int32_t(blocks);
    info.flattened = flat && c.rows > 1;
    info.path = 1;
    info.vector_units = p.units;
    info.tail_elems = p.tail_units;
    t_last_launch = info;
    return GLU_OK;
}

void mark_noop()
{
    t_last_launch = glu_launch_info_t{};
}

}  // namespace

namespace glu {

int cuda_fail(cudaError_t e)
{
    snprintf(t_cuda_error, sizeof(t_cuda_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return GLU_ERR_CUDA;
}

int validate_fwd(const void *a, int64_t a_stride, const void *b, int64_t b_stride, const void *y,
                 int64_t y_stride, int64_t n_rows, int64_t n_cols, int layout, int act, int dtype,
                 Call *c)
{
    *c = Call{};
    if (!valid_enums(layout, act, dtype)) return GLU_ERR_ENUM;
    if (n_rows < 0 || n_cols < 0) return GLU_ERR_SHAPE;
    if (n_rows == 0 || n_cols == 0) { c->empty = true; return GLU_OK; }
    const bool concat = layout == GLU_LAYOUT_CONCAT;
    if (!a || !y || (!concat && !b)) return GLU_ERR_NULL;
    const int E = elem_size(dtype);
    if (n_rows == 1) { a_stride = concat ? 2 * n_cols : n_cols; b_stride = n_cols; y_stride = n_cols; }
    if (concat) {
        if (n_cols > INT64_MAX / 2) return GLU_ERR_SHAPE;
        if (a_stride < 2 * n_cols) return GLU_ERR_STRIDE;
        if (uintptr_t(a) > UINTPTR_MAX - uintptr_t(n_cols) * E) return GLU_ERR_SHAPE;
        b = static_cast<const char *>(a) + n_cols * E;
        b_stride = a_stride;
    } else if (a_stride < n_cols || b_stride < n_cols) {
        return GLU_ERR_STRIDE;
    }
    if (y_stride < n_cols) return GLU_ERR_STRIDE;

    const Mat ma{uintptr_t(a), a_stride, n_cols}, mb{uintptr_t(b), b_stride, n_cols};
    const Mat my{uintptr_t(y), y_stride, n_cols};
    const Mat mx{uintptr_t(a), a_stride, concat ? 2 * n_cols : n_cols};
    if (extent_bytes(mx, n_rows, E) < 0 || extent_bytes(mb, n_rows, E) < 0 ||
        extent_bytes(my, n_rows, E) < 0)
        return GLU_ERR_SHAPE;
    const Mat ins[2] = {ma, mb};
    if (int st = check_aliasing(ins, 2, &my, 1, n_rows, E)) return st;

    c->dir = kFwd; c->act = act; c->dtype = dtype; c->E = E;
    c->rows = n_rows; c->cols = n_cols;
    c->a = static_cast<const char *>(a); c->b = static_cast<const char *>(b);
    c->y0 = static_cast<char *>(const_cast<void *>(y));
    c->sa = a_stride; c->sb = b_stride; c->sy0 = y_stride;
    return GLU_OK;
}

int validate_add_rmsnorm(const void *x, int64_t x_stride, const void *res, int64_t res_stride,
                         const void *gamma, const void *h, int64_t h_stride, const void *y, int64_t y_stride,
                         const float *rstd, int64_t n_rows, int64_t n_cols, float eps, int dtype, bool *empty)
{
    *empty = false;
    if (!(dtype == GLU_F32 || dtype == GLU_F16 || dtype == GLU_BF16)) return GLU_ERR_ENUM;
    if (n_rows < 0 || n_cols < 0) return GLU_ERR_SHAPE;
    if (!(eps > 0.0f) || !(eps < INFINITY)) return GLU_ERR_VALUE;
    if (n_rows == 0 || n_cols == 0) { *empty = true; return GLU_OK; }
    if (n_cols > kRmsMaxCols) return GLU_ERR_SHAPE;
    if (!x || !res || !gamma || !h || !y) return GLU_ERR_NULL;
    if (n_rows == 1) x_stride = res_stride = h_stride = y_stride = n_cols;
    if (x_stride < n_cols || res_stride < n_cols || h_stride < n_cols || y_stride < n_cols)
        return GLU_ERR_STRIDE;
    const int E = elem_size(dtype);
    const Mat mx{uintptr_t(x), x_stride, n_cols}, mr{uintptr_t(res), res_stride, n_cols};
    const Mat mh{uintptr_t(h), h_stride, n_cols}, my{uintptr_t(y), y_stride, n_cols};
    const Mat mg{uintptr_t(gamma), n_cols, n_cols};
    if (extent_bytes(mx, n_rows, E) < 0 || extent_bytes(mr, n_rows, E) < 0 || extent_bytes(mh, n_rows, E) < 0 ||
        extent_bytes(my, n_rows, E) < 0 || extent_bytes(mg, 1, E) < 0)
        return GLU_ERR_SHAPE;
    const Mat ins[2] = {mx, mr}, outs[2] = {mh, my};
    if (int st = check_aliasing(ins, 2, outs, 2, n_rows, E)) return st;
    // gamma is read by every row: no output element may lie on it
    for (const Mat &o : outs)
        if (rows_hit_range(o, n_rows, E, mg.p, uint64_t(n_cols) * E)) return GLU_ERR_ALIAS;
    if (rstd) {
        if (uint64_t(n_rows) > (UINTPTR_MAX - uintptr_t(rstd)) / 4) return GLU_ERR_SHAPE;
        const uint64_t r0 = uintptr_t(rstd), r1 = r0 + uint64_t(n_rows) * 4;
        const Mat all[5] = {mx, mr, mh, my, mg};
        for (int k = 0; k < 5; ++k) {
            const uint64_t a0 = all[k].p, a1 = a0 + uint64_t(extent_bytes(all[k], k == 4 ? 1 : n_rows, E));
            if (!(a1 <= r0 || r1 <= a0)) return GLU_ERR_ALIAS;
        }
    }
    return GLU_OK;
}

int validate_add_rmsnorm_bwd(const void *dy, int64_t dy_stride, const void *h, int64_t h_stride, const float *rstd,
                             const void *gamma, const void *dh, int64_t dh_stride, const void *dx, int64_t dx_stride,
                             const void *dres, int64_t dres_stride, const float *dgamma, int64_t n_rows,
                             int64_t n_cols, int dtype, bool *empty)
{
    *empty = false;
    if (!(dtype == GLU_F32 || dtype == GLU_F16 || dtype == GLU_BF16)) return GLU_ERR_ENUM;
    if (n_rows < 0 || n_cols < 0) return GLU_ERR_SHAPE;
    if (n_rows == 0 || n_cols == 0) { *empty = true; return GLU_OK; }
    if (n_cols > kRmsBwdMaxCols) return GLU_ERR_SHAPE;
    if (!dy || !h || !rstd || !gamma || !dx) return GLU_ERR_NULL;
    if (n_rows == 1) dy_stride = h_stride = dh_stride = dx_stride = dres_stride = n_cols;
    if (dy_stride < n_cols || h_stride < n_cols || dx_stride < n_cols || (dh && dh_stride < n_cols) ||
        (dres && dres_stride < n_cols))
        return GLU_ERR_STRIDE;
    const int E = elem_size(dtype);
    const Mat mdy{uintptr_t(dy), dy_stride, n_cols}, mh{uintptr_t(h), h_stride, n_cols};
    const Mat mdh{uintptr_t(dh), dh_stride, n_cols}, mdx{uintptr_t(dx), dx_stride, n_cols};
    const Mat mdr{uintptr_t(dres), dres_stride, n_cols}, mg{uintptr_t(gamma), n_cols, n_cols};
    if (extent_bytes(mdy, n_rows, E) < 0 || extent_bytes(mh, n_rows, E) < 0 || extent_bytes(mdx, n_rows, E) < 0 ||
        (dh && extent_bytes(mdh, n_rows, E) < 0) || (dres && extent_bytes(mdr, n_rows, E) < 0) ||
        extent_bytes(mg, 1, E) < 0)
        return GLU_ERR_SHAPE;
    Mat ins[3] = {mdy, mh, mdh}, outs[2] = {mdx, mdr};
    if (int st = check_aliasing(ins, dh ? 3 : 2, outs, dres ? 2 : 1, n_rows, E)) return st;
    // small read-only and accumulated vectors: no matrix output may touch them
    // and they may not touch each other or any matrix
    const uint64_t gb = uint64_t(n_cols) * E, rb = uint64_t(n_rows) * 4, db = uint64_t(n_cols) * 4;
    if (uint64_t(n_rows) > (UINTPTR_MAX - uintptr_t(rstd)) / 4) return GLU_ERR_SHAPE;
    if (dgamma && uint64_t(n_cols) > (UINTPTR_MAX - uintptr_t(dgamma)) / 4) return GLU_ERR_SHAPE;
    for (int o = 0; o < (dres ? 2 : 1); ++o)
        if (rows_hit_range(outs[o], n_rows, E, mg.p, gb) || rows_hit_range(outs[o], n_rows, E, uintptr_t(rstd), rb) ||
            (dgamma && rows_hit_range(outs[o], n_rows, E, uintptr_t(dgamma), db)))
            return GLU_ERR_ALIAS;
    if (dgamma) {
        const Mat all[5] = {mdy, mh, mdh, mdx, mdr};
        for (int k = 0; k < 5; ++k) {
            if ((k == 2 && !dh) || (k == 4 && !dres)) continue;
            if (rows_hit_range(all[k], n_rows, E, uintptr_t(dgamma), db)) return GLU_ERR_ALIAS;
        }
        const uint64_t d0 = uintptr_t(dgamma), g0 = mg.p, r0 = uintptr_t(rstd);
        if (!(d0 + db <= g0 || g0 + gb <= d0) || !(d0 + db <= r0 || r0 + rb <= d0)) return GLU_ERR_ALIAS;
    }
    return GLU_OK;
}

int validate_bwd(const void *dc, int64_t dc_stride, const void *a, int64_t a_stride, const void *b,
                 int64_t b_stride, const void *da, int64_t da_stride, const void *db,
                 int64_t db_stride, int64_t n_rows, int64_t n_cols, int layout, int act, int dtype,
                 Call *c)
{
    *c = Call{};
    if (!valid_enums(layout, act, dtype)) return GLU_ERR_ENUM;
    if (n_rows < 0 || n_cols < 0) return GLU_ERR_SHAPE;
    if (n_rows == 0 || n_cols == 0) { c->empty = true; return GLU_OK; }
    const bool concat = layout == GLU_LAYOUT_CONCAT;
    if (!dc || !a || !da || (!concat && (!b || !db))) return GLU_ERR_NULL;
    const int E = elem_size(dtype);
    if (n_rows == 1) {
        dc_stride = n_cols;
        a_stride = da_stride = concat ? 2 * n_cols : n_cols;
        b_stride = db_stride = n_cols;
    }
    if (concat) {
        if (n_cols > INT64_MAX / 2) return GLU_ERR_SHAPE;
        if (a_stride < 2 * n_cols || da_stride < 2 * n_cols) return GLU_ERR_STRIDE;
        if (uintptr_t(a) > UINTPTR_MAX - uintptr_t(n_cols) * E ||
            uintptr_t(da) > UINTPTR_MAX - uintptr_t(n_cols) * E)
            return GLU_ERR_SHAPE;
        b = static_cast<const char *>(a) + n_cols * E;
        b_stride = a_stride;
        db = static_cast<const char *>(da) + n_cols * E;
        db_stride = da_stride;
    } else if (a_stride < n_cols || b_stride < n_cols || da_stride < n_cols || db_stride < n_cols) {
        return GLU_ERR_STRIDE;
    }
    if (dc_stride < n_cols) return GLU_ERR_STRIDE;

    const Mat mc{uintptr_t(dc), dc_stride, n_cols};
    const Mat ma{uintptr_t(a), a_stride, n_cols}, mb{uintptr_t(b), b_stride, n_cols};
    const Mat mda{uintptr_t(da), da_stride, n_cols}, mdb{uintptr_t(db), db_stride, n_cols};
    const Mat mx{uintptr_t(a), a_stride, concat ? 2 * n_cols : n_cols};
    const Mat mdx{uintptr_t(da), da_stride, concat ? 2 * n_cols : n_cols};
    if (extent_bytes(mc, n_rows, E) < 0 || extent_bytes(mx, n_rows, E) < 0 ||
        extent_bytes(mb, n_rows, E) < 0 || extent_bytes(mdx, n_rows, E) < 0 ||
        extent_bytes(mdb, n_rows, E) < 0)
        return GLU_ERR_SHAPE;
    const Mat ins[3] = {mc, ma, mb};
    const Mat outs[2] = {mda, mdb};
    if (int st = check_aliasing(ins, 3, outs, 2, n_rows, E)) return st;

    c->dir = kBwd; c->act = act; c->dtype = dtype; c->E = E;
    c->rows = n_rows; c->cols = n_cols;
    c->a = static_cast<const char *>(a); c->b = static_cast<const char *>(b);
    c->dc = static_cast<const char *>(dc);
    c->y0 = static_cast<char *>(const_cast<void *>(da));
    c->y1 = static_cast<char *>(const_cast<void *>(db));
    c->sa = a_stride; c->sb = b_stride; c->sdc = dc_stride; c->sy0 = da_stride; c->sy1 = db_stride;
    return GLU_OK;
}

}  // namespace glu

namespace glu {
void record_launch(const glu_launch_info_t &info) { t_last_launch = info; }

// Waits of the self-test kernel that ran out (each launch should add one).
static __device__ unsigned int g_selftest_timeouts;

// One warp waits on a shared-memory barrier that nothing arrives on, with the
// bounded, sleeping wait the staged kernels use: the wait must run out and
// the kernel return.
__global__ void wait_selftest_kernel()
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    const bool completed = __any_sync(0xFFFFFFFFu, mbar_wait_sleep(smem_u32(&bar), 0));
    if (threadIdx.x == 0 && !completed) atomicAdd(&g_selftest_timeouts, 1u);
}

cudaError_t on_device(const void *p, bool *yes)
{
    cudaPointerAttributes a{};
    const cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return e;
    }
    *yes = a.type == cudaMemoryTypeDevice;
    return cudaSuccess;
}
}  // namespace glu

extern "C" {

int glu_fwd(const void *a, int64_t a_stride, const void *b, int64_t b_stride, void *y,
            int64_t y_stride, int64_t n_rows, int64_t n_cols, glu_layout_t layout,
            glu_act_t act, glu_dtype_t dtype, glu_stream_t stream)
{
    Call c;
    const int st = glu::validate_fwd(a, a_stride, b, b_stride, y, y_stride, n_rows, n_cols, layout,
                                     act, dtype, &c);
    if (st != GLU_OK) return st;
    if (c.empty) { mark_noop(); return GLU_OK; }
    return plan_and_launch(c, reinterpret_cast<cudaStream_t>(stream));
}

int glu_bwd(const void *dc, int64_t dc_stride, const void *a, int64_t a_stride, const void *b,
            int64_t b_stride, void *da, int64_t da_stride, void *db, int64_t db_stride,
            int64_t n_rows, int64_t n_cols, glu_layout_t layout, glu_act_t act,
            glu_dtype_t dtype, glu_stream_t stream)
{
    Call c;
    const int st = glu::validate_bwd(dc, dc_stride, a, a_stride, b, b_stride, da, da_stride, db,
                                     db_stride, n_rows, n_cols, layout, act, dtype, &c);
    if (st != GLU_OK) return st;
    if (c.empty) { mark_noop(); return GLU_OK; }
    return plan_and_launch(c, reinterpret_cast<cudaStream_t>(stream));
}

const char *glu_status_string(int status)
{
    switch (status) {
    case GLU_OK: return "ok";
    case GLU_ERR_NULL: return "a required pointer is NULL";
    case GLU_ERR_SHAPE: return "negative size, or a size whose byte extent overflows";
    case GLU_ERR_STRIDE: return "a row stride is smaller than its row width";
    case GLU_ERR_ALIAS: return "an output overlaps an input other than exactly, or another output";
    case GLU_ERR_ENUM: return "unknown activation, layout, dtype or tuning value";
    case GLU_ERR_CUDA: return "the CUDA runtime refused a launch or copy";
    case GLU_ERR_WORKSPACE: return "the workspace is NULL or too small for one row";
    case GLU_ERR_VALUE:
        return "an argument is out of range (eps not finite and > 0, or a GEMM operand or dgamma not in device "
               "memory)";
    default: return "unknown status";
    }
}

const char *glu_last_cuda_error(void) { return t_cuda_error; }

int glu_version(void) { return GLU_VERSION; }

int glu_wait_timeouts(unsigned int *count, int reset)
{
    if (!count) return GLU_ERR_NULL;
    unsigned int bulk = 0, gemm = 0, rms = 0, self = 0;
    cudaError_t e = glu::bulk_timeouts(&bulk, reset != 0);
    if (e == cudaSuccess) e = glu::gemm::timeouts(&gemm, reset != 0);
    if (e == cudaSuccess) e = glu::rms::timeouts(&rms, reset != 0);
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&self, glu::g_selftest_timeouts, sizeof(unsigned int));
    if (e == cudaSuccess && reset) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(glu::g_selftest_timeouts, &zero, sizeof(unsigned int));
    }
    if (e != cudaSuccess) return cuda_fail(e);
    *count = bulk + gemm + rms + self;
    return GLU_OK;
}

int glu_wait_selftest(glu_stream_t stream)
{
    glu::wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>();
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    glu_launch_info_t info{};
    info.launched = 1;
    info.threads = 32;
    info.grid = 1;
    glu::record_launch(info);
    return GLU_OK;
}

int glu_last_launch(glu_launch_info_t *out)
{
    if (!out) return GLU_ERR_NULL;
    *out = t_last_launch;
    return GLU_OK;
}

int glu_set_tuning(const glu_tuning_t *t)
{
    if (!t) return GLU_ERR_NULL;
    const int32_t v = t->vec_bytes, u = t->unroll, c = t->ctas_per_sm, d = t->dependent_launch;
    const int32_t path = t->path;
    if (path < 0 || path > 2) return GLU_ERR_ENUM;
    if (!(v == 0 || v == 32 || v == 16 || v == 4 || v == 2)) return GLU_ERR_ENUM;
    if (!(u == 0 || u == 1 || u == 2 || u == 4)) return GLU_ERR_ENUM;
    if (c > 64) return GLU_ERR_ENUM;
    if (d < -1 || d > 1) return GLU_ERR_ENUM;
    g_vec_bytes.store(v);
    g_unroll.store(u);
    g_ctas_per_sm.store(c);
    g_dependent_launch.store(d);
    g_path.store(path);
    return GLU_OK;
}

int glu_get_tuning(glu_tuning_t *out)
{
    if (!out) return GLU_ERR_NULL;
    out->vec_bytes = g_vec_bytes.load();
    out->unroll = g_unroll.load();
    out->ctas_per_sm = g_ctas_per_sm.load();
    out->dependent_launch = g_dependent_launch.load();
    out->path = g_path.load();
    return GLU_OK;
}

}  // extern "C"
