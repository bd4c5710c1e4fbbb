// Host-memory entry points (glu_fwd_host, glu_bwd_host, glu_host_workspace_bytes):
// the operands live in host memory; blocks of rows are copied into a device
// workspace the caller supplies, processed by the same kernels as glu_fwd /
// glu_bwd, and copied back.  Two workspace slots alternate, so that while the
// kernels work on one block the next block's inputs are already on their way
// in and the previous block's outputs on their way out.  Contracts are in
// include/glu.h.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

#include "glu.h"
#include "glu_internal.h"

namespace {

constexpr int kSlots = 2;
constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int elem_size(int dtype) { return dtype == GLU_F32 ? 4 : 2; }

bool valid_enums(int layout, int act, int dtype)
{
    return (layout == GLU_LAYOUT_SPLIT || layout == GLU_LAYOUT_CONCAT) &&
           (act >= GLU_ACT_SILU && act <= GLU_ACT_RELU) &&
           (dtype == GLU_F32 || dtype == GLU_F16 || dtype == GLU_BF16);
}

// The staged matrices of one slot, by direction and layout, as row widths in
// elements: inputs first, then outputs.
struct SlotShape {
    int n_in, n_out;
    int64_t width[5];
};

SlotShape slot_shape(int backward, int layout, int64_t C)
{
    const bool concat = layout == GLU_LAYOUT_CONCAT;
    if (!backward) {
        if (concat) return {1, 1, {2 * C, C}};                 // x | y
        return {2, 1, {C, C, C}};                               // a, b | y
    }
    if (concat) return {2, 1, {C, 2 * C, 2 * C}};               // dc, x | dx
    return {3, 2, {C, C, C, C, C}};                             // dc, a, b | da, db
}

// Workspace bytes for two slots of `rows` rows; 0 on overflow.
size_t workspace_for(const SlotShape &sh, int64_t rows, int E)
{
    size_t slot = 0;
    for (int m = 0; m < sh.n_in + sh.n_out; ++m) {
        const double approx = double(rows) * double(sh.width[m]) * E;
        if (approx > 1e18) return 0;
        slot += round_up(size_t(rows) * size_t(sh.width[m]) * size_t(E));
    }
    return kSlots * slot;
}

// Largest number of rows whose two slots fit in `bytes`.
int64_t rows_that_fit(const SlotShape &sh, size_t bytes, int E, int64_t n_rows)
{
    size_t per_row = 0;
    for (int m = 0; m < sh.n_in + sh.n_out; ++m) per_row += size_t(sh.width[m]) * E;
    const size_t pad = size_t(sh.n_in + sh.n_out) * kAlign;
    if (bytes / kSlots <= pad) return 0;
    int64_t r = int64_t((bytes / kSlots - pad) / per_row);
    if (r > n_rows) r = n_rows;
    while (r > 0 && workspace_for(sh, r, E) > bytes) --r;
    return r;
}

struct Host {
    const char *p;     // base (host)
    int64_t stride;    // elements
    int64_t width;     // elements per row
};

// Rows [r0, r0 + rows) of a host matrix <-> a packed device block.
cudaError_t copy_rows(void *dev, const Host &h, int64_t r0, int64_t rows, int E, bool to_device,
                      cudaStream_t s)
{
    const size_t row_bytes = size_t(h.width) * E;
    char *hp = const_cast<char *>(h.p) + size_t(r0) * size_t(h.stride) * E;
    if (rows == 1 || h.stride == h.width) {
        const size_t n = row_bytes * size_t(rows);
        return to_device ? cudaMemcpyAsync(dev, hp, n, cudaMemcpyHostToDevice, s)
                         : cudaMemcpyAsync(hp, dev, n, cudaMemcpyDeviceToHost, s);
    }
    const size_t pitch = size_t(h.stride) * E;
    return to_device ? cudaMemcpy2DAsync(dev, row_bytes, hp, pitch, row_bytes, size_t(rows),
                                         cudaMemcpyHostToDevice, s)
                     : cudaMemcpy2DAsync(hp, pitch, dev, row_bytes, row_bytes, size_t(rows),
                                         cudaMemcpyDeviceToHost, s);
}

using glu::cuda_fail;

// The pipeline shared by both directions.  `in`/`out` are the host matrices
// in slot order; `launch` runs the kernel of one block on device pointers.
template <class Launch>
int run_pipeline(const SlotShape &sh, const Host *in, const Host *out, int64_t n_rows, int E,
                 void *workspace, size_t workspace_bytes, cudaStream_t s_in, cudaStream_t s_k,
                 cudaStream_t s_out, Launch launch)
{
    const int64_t chunk = rows_that_fit(sh, workspace_bytes, E, n_rows);
    if (chunk < 1) return GLU_ERR_WORKSPACE;

    // slot s, matrix m -> device address
    char *dev[kSlots][5];
    {
        char *p = static_cast<char *>(workspace);
        for (int s = 0; s < kSlots; ++s)
            for (int m = 0; m < sh.n_in + sh.n_out; ++m) {
                dev[s][m] = p;
                p += round_up(size_t(chunk) * size_t(sh.width[m]) * size_t(E));
            }
    }

    cudaEvent_t entry = nullptr, in_ready[kSlots] = {}, k_done[kSlots] = {}, out_done[kSlots] = {};
    cudaError_t e = cudaEventCreateWithFlags(&entry, cudaEventDisableTiming);
    for (int s = 0; s < kSlots && e == cudaSuccess; ++s) {
        e = cudaEventCreateWithFlags(&in_ready[s], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&k_done[s], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&out_done[s], cudaEventDisableTiming);
    }
    int status = GLU_OK;
    auto check = [&](cudaError_t err) {
        if (err != cudaSuccess && status == GLU_OK) status = cuda_fail(err);
        return status == GLU_OK;
    };
    if (!check(e)) goto cleanup;

    // the copy streams start after everything already enqueued on the compute stream
    if (!check(cudaEventRecord(entry, s_k))) goto cleanup;
    if (!check(cudaStreamWaitEvent(s_in, entry, 0))) goto cleanup;
    if (!check(cudaStreamWaitEvent(s_out, entry, 0))) goto cleanup;

    for (int64_t r0 = 0, i = 0; r0 < n_rows; r0 += chunk, ++i) {
        const int s = int(i % kSlots);
        const int64_t rows = n_rows - r0 < chunk ? n_rows - r0 : chunk;
        // inputs of block i go where block i - 2's inputs were: wait for its kernel
        if (i >= kSlots && !check(cudaStreamWaitEvent(s_in, k_done[s], 0))) goto cleanup;
        for (int m = 0; m < sh.n_in; ++m)
            if (!check(copy_rows(dev[s][m], in[m], r0, rows, E, true, s_in))) goto cleanup;
        if (!check(cudaEventRecord(in_ready[s], s_in))) goto cleanup;
        // the kernel needs its inputs, and block i - 2's outputs must be out of the slot
        if (!check(cudaStreamWaitEvent(s_k, in_ready[s], 0))) goto cleanup;
        if (i >= kSlots && !check(cudaStreamWaitEvent(s_k, out_done[s], 0))) goto cleanup;
        const int st = launch(dev[s], rows, s_k);
        if (st != GLU_OK) { status = st; goto cleanup; }
        if (!check(cudaEventRecord(k_done[s], s_k))) goto cleanup;
        if (!check(cudaStreamWaitEvent(s_out, k_done[s], 0))) goto cleanup;
        for (int m = 0; m < sh.n_out; ++m)
            if (!check(copy_rows(dev[s][sh.n_in + m], out[m], r0, rows, E, false, s_out))) goto cleanup;
        if (!check(cudaEventRecord(out_done[s], s_out))) goto cleanup;
    }
    // work enqueued later on the compute stream runs after the last copy-out
    {
        const int last = int(((n_rows + chunk - 1) / chunk - 1) % kSlots);
        check(cudaStreamWaitEvent(s_k, out_done[last], 0));
    }

cleanup:
    // destroying an event with work pending on it is allowed: its resources are
    // released once that work completes
    if (entry) cudaEventDestroy(entry);
    for (int s = 0; s < kSlots; ++s) {
        if (in_ready[s]) cudaEventDestroy(in_ready[s]);
        if (k_done[s]) cudaEventDestroy(k_done[s]);
        if (out_done[s]) cudaEventDestroy(out_done[s]);
    }
    return status;
}

}  // namespace

extern "C" {

size_t glu_host_workspace_bytes(int64_t rows_per_block, int64_t n_cols, glu_layout_t layout,
                                glu_dtype_t dtype, int backward)
{
    if (!valid_enums(layout, GLU_ACT_SILU, dtype) || rows_per_block < 1 || n_cols < 1) return 0;
    return workspace_for(slot_shape(backward != 0, layout, n_cols), rows_per_block, elem_size(dtype));
}

int glu_fwd_host(const void *a, int64_t a_stride, const void *b, int64_t b_stride, void *y,
                 int64_t y_stride, int64_t n_rows, int64_t n_cols, glu_layout_t layout,
                 glu_act_t act, glu_dtype_t dtype, void *workspace, size_t workspace_bytes,
                 glu_stream_t copy_in, glu_stream_t compute, glu_stream_t copy_out)
{
    // the host matrices obey glu_fwd's rules (shapes, strides, NULLs, aliasing)
    glu::Call c;
    const int pre = glu::validate_fwd(a, a_stride, b, b_stride, y, y_stride, n_rows, n_cols, layout,
                                      act, dtype, &c);
    if (pre != GLU_OK || c.empty) return pre;
    if (!workspace) return GLU_ERR_WORKSPACE;
    const bool concat = layout == GLU_LAYOUT_CONCAT;
    const int E = c.E;
    const SlotShape sh = slot_shape(0, layout, n_cols);
    Host in[2], out[1];
    if (concat) {
        in[0] = {c.a, c.sa, 2 * n_cols};
    } else {
        in[0] = {c.a, c.sa, n_cols};
        in[1] = {c.b, c.sb, n_cols};
    }
    out[0] = {c.y0, c.sy0, n_cols};
    // Each block's inputs are copied in before its outputs are copied out and
    // blocks are disjoint row ranges, so an output that is exactly an input
    // (in place) is read before it is overwritten.
    auto launch = [&](char *const *d, int64_t rows, cudaStream_t s) {
        if (concat)
            return glu_fwd(d[0], 2 * n_cols, nullptr, 0, d[1], n_cols, rows, n_cols, layout, act, dtype,
                           reinterpret_cast<glu_stream_t>(s));
        return glu_fwd(d[0], n_cols, d[1], n_cols, d[2], n_cols, rows, n_cols, layout, act, dtype,
                       reinterpret_cast<glu_stream_t>(s));
    };
    return run_pipeline(sh, in, out, n_rows, E, workspace, workspace_bytes,
                        reinterpret_cast<cudaStream_t>(copy_in), reinterpret_cast<cudaStream_t>(compute),
                        reinterpret_cast<cudaStream_t>(copy_out), launch);
}

int glu_bwd_host(const void *dc, int64_t dc_stride, const void *a, int64_t a_stride, const void *b,
                 int64_t b_stride, void *da, int64_t da_stride, void *db, int64_t db_stride,
                 int64_t n_rows, int64_t n_cols, glu_layout_t layout, glu_act_t act, glu_dtype_t dtype,
                 void *workspace, size_t workspace_bytes, glu_stream_t copy_in, glu_stream_t compute,
                 glu_stream_t copy_out)
{
    glu::Call c;
    const int pre = glu::validate_bwd(dc, dc_stride, a, a_stride, b, b_stride, da, da_stride, db,
                                      db_stride, n_rows, n_cols, layout, act, dtype, &c);
    if (pre != GLU_OK || c.empty) return pre;
    if (!workspace) return GLU_ERR_WORKSPACE;
    const bool concat = layout == GLU_LAYOUT_CONCAT;
    const int E = c.E;
    const SlotShape sh = slot_shape(1, layout, n_cols);
    Host in[3], out[2];
    in[0] = {c.dc, c.sdc, n_cols};
    if (concat) {
        in[1] = {c.a, c.sa, 2 * n_cols};
        out[0] = {c.y0, c.sy0, 2 * n_cols};
    } else {
        in[1] = {c.a, c.sa, n_cols};
        in[2] = {c.b, c.sb, n_cols};
        out[0] = {c.y0, c.sy0, n_cols};
        out[1] = {c.y1, c.sy1, n_cols};
    }
    auto launch = [&](char *const *d, int64_t rows, cudaStream_t s) {
        if (concat)
            return glu_bwd(d[0], n_cols, d[1], 2 * n_cols, nullptr, 0, d[2], 2 * n_cols, nullptr, 0, rows,
                           n_cols, layout, act, dtype, reinterpret_cast<glu_stream_t>(s));
        return glu_bwd(d[0], n_cols, d[1], n_cols, d[2], n_cols, d[3], n_cols, d[4], n_cols, rows, n_cols,
                       layout, act, dtype, reinterpret_cast<glu_stream_t>(s));
    };
    return run_pipeline(sh, in, out, n_rows, E, workspace, workspace_bytes,
                        reinterpret_cast<cudaStream_t>(copy_in), reinterpret_cast<cudaStream_t>(compute),
                        reinterpret_cast<cudaStream_t>(copy_out), launch);
}

}  // extern "C"
