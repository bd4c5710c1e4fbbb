// glu_fwd_host_noalloc: the host-memory forward (the operation of
// glu_fwd_host) for callers that cannot allocate device memory at all.
//
// glu_fwd_host needs a device workspace from its caller.  Some callers cannot
// provide one: a plug-in running inside a host application whose own allocator
// owns all device memory and hands none out, or a process that fixes its memory
// budget at start-up and must not allocate once it is running.  This entry
// point stages the blocks of rows in a fixed array that lives inside the
// library instead, so the caller passes only the host inputs and outputs.
//
// The array is a file-scope device variable of GLU_NOALLOC_SCRATCH_BYTES
// (32 MiB): every GPU on which the library's module is loaded holds it until
// the process exits.  Its name in host code is only a stand-in for the device
// variable, so the host looks up its device address once per device with
// cudaGetSymbolAddress and hands that address to the copies and kernels.
// Nothing in the array has to start at zero: each block's inputs are copied in
// before the kernel reads them, and the kernel writes every output element
// before it is copied out.  Every call shares the array, so calls whose work
// overlaps on the GPU (on different streams, or from different threads without
// ordering) race on it.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "glu.h"
#include "glu_internal.h"

namespace {

constexpr size_t kScratchBytes = GLU_NOALLOC_SCRATCH_BYTES;
constexpr size_t kAlign = 256;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch_addr[kMaxDevices];
std::mutex g_setup_mutex;

// Device address of g_noalloc_scratch on the current device, looked up on the
// first call made on that device (devices numbered kMaxDevices and above are
// looked up on every call).  *dev_out receives the device number.
int scratch_address(void **out, int *dev_out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return glu::cuda_fail(e);
    *dev_out = dev;
    if (dev < 0) return glu::cuda_fail(cudaErrorInvalidDevice);
    if (dev >= kMaxDevices) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) return glu::cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
        *out = p;
        return GLU_OK;
    }
    void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        p = g_scratch_addr[dev].load(std::memory_order_acquire);
        if (!p) {
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || !p) return glu::cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
            g_scratch_addr[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return GLU_OK;
}

// A failed copy may mean the cached address is stale (the device was reset,
// which reloads the library's module): the next call looks it up again.
int forget_address(int dev, cudaError_t e)
{
    if (dev >= 0 && dev < kMaxDevices) g_scratch_addr[dev].store(nullptr, std::memory_order_release);
    return glu::cuda_fail(e);
}

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Rows [r0, r0 + rows) of a host matrix <-> a packed device block, on `s`.
cudaError_t stage_rows(void *dev, const char *host, int64_t stride, int64_t width, int64_t r0, int64_t rows,
                       int E, bool to_device, cudaStream_t s)
{
    const size_t row_bytes = size_t(width) * E;
    char *hp = const_cast<char *>(host) + size_t(r0) * size_t(stride) * E;
    if (rows == 1 || stride == width) {
        const size_t n = row_bytes * size_t(rows);
        return to_device ? cudaMemcpyAsync(dev, hp, n, cudaMemcpyHostToDevice, s)
                         : cudaMemcpyAsync(hp, dev, n, cudaMemcpyDeviceToHost, s);
    }
    const size_t pitch = size_t(stride) * E;
    return to_device ? cudaMemcpy2DAsync(dev, row_bytes, hp, pitch, row_bytes, size_t(rows),
                                         cudaMemcpyHostToDevice, s)
                     : cudaMemcpy2DAsync(hp, pitch, dev, row_bytes, row_bytes, size_t(rows),
                                         cudaMemcpyDeviceToHost, s);
}

}  // namespace

extern "C" int glu_fwd_host_noalloc(const void *a, int64_t a_stride, const void *b, int64_t b_stride,
                                    void *y, int64_t y_stride, int64_t n_rows, int64_t n_cols,
                                    glu_layout_t layout, glu_act_t act, glu_dtype_t dtype,
                                    glu_stream_t stream)
{
    glu::Call c;
    const int pre = glu::validate_fwd(a, a_stride, b, b_stride, y, y_stride, n_rows, n_cols, layout, act,
                                      dtype, &c);
    if (pre != GLU_OK || c.empty) return pre;
    const bool concat = layout == GLU_LAYOUT_CONCAT;
    const int E = c.E;

    // One block of rows at a time: [inputs | output] packed in the array.
    const int64_t in_width = concat ? 2 * n_cols : n_cols;    // x, or each of a and b
    const int n_in = concat ? 1 : 2;
    const size_t row_bytes = size_t(n_in) * size_t(in_width) * E + size_t(n_cols) * E;
    const size_t pad = size_t(n_in + 1) * kAlign;
    if (row_bytes > kScratchBytes || kScratchBytes - pad < row_bytes) return GLU_ERR_WORKSPACE;
    int64_t block = int64_t((kScratchBytes - pad) / row_bytes);
    if (block > n_rows) block = n_rows;

    void *base = nullptr;
    int dev = -1;
    if (int st = scratch_address(&base, &dev)) return st;
    char *d_in[2], *d_out;
    {
        char *p = static_cast<char *>(base);
        for (int m = 0; m < n_in; ++m) {
            d_in[m] = p;
            p += round_up(size_t(block) * size_t(in_width) * E);
        }
        d_out = p;
    }

    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const char *h_in[2] = {c.a, c.b};
    const int64_t h_stride[2] = {c.sa, c.sb};
    for (int64_t r0 = 0; r0 < n_rows; r0 += block) {
        const int64_t rows = n_rows - r0 < block ? n_rows - r0 : block;
        for (int m = 0; m < n_in; ++m) {
            cudaError_t e = stage_rows(d_in[m], h_in[m], h_stride[m], in_width, r0, rows, E, true, s);
            if (e != cudaSuccess) return forget_address(dev, e);
        }
        const int st = concat ? glu_fwd(d_in[0], 2 * n_cols, nullptr, 0, d_out, n_cols, rows, n_cols, layout,
                                        act, dtype, stream)
                              : glu_fwd(d_in[0], n_cols, d_in[1], n_cols, d_out, n_cols, rows, n_cols, layout,
                                        act, dtype, stream);
        if (st != GLU_OK) return st;
        cudaError_t e = stage_rows(d_out, c.y0, c.sy0, n_cols, r0, rows, E, false, s);
        if (e != cudaSuccess) return forget_address(dev, e);
    }
    return GLU_OK;
}
