// Declarations shared by the library's host-side translation units: argument
// validation, error recording, the bulk-copy and GEMM timeout counters and the
// per-thread launch record.  The streaming kernels' own layout is glu_plan.h.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "glu.h"
#include "glu_plan.h"

namespace glu {


// Bulk-copy staging kernels (glu_bulk.cu): contiguous operands only, one
// ("wide") or two ("narrow") blocks per SM, `chunks` chunks of kBulkChunkHost
// bytes per operand.
struct BulkParams {
    const char *a, *b, *dc;        // inputs (dc: backward only)
    char *y0, *y1;                 // outputs (y1: backward only)
    int64_t chunks;                // whole chunks of kBulkChunkHost bytes per operand
};
using BulkFn = void (*)(BulkParams);
constexpr int kBulkChunkHost = 16384;
BulkFn bulk_kernel(int dtype, int act, int dir, bool narrow);
int bulk_smem_bytes(int dir, bool narrow);
int bulk_threads(bool narrow);
cudaError_t bulk_timeouts(unsigned int *count, bool reset);
namespace gemm {
cudaError_t timeouts(unsigned int *count, bool reset);   // glu_gemm.cu
}
namespace rms {
cudaError_t timeouts(unsigned int *count, bool reset);   // glu_rmsnorm.cu
}
void record_launch(const glu_launch_info_t &info);       // this thread's glu_last_launch
// Whether p points into device memory (not pinned host or managed memory):
// the tensor-memory accelerator and the bulk-copy engine are given device
// memory only.
cudaError_t on_device(const void *p, bool *yes);

// Fused residual add + RMSNorm (glu_rmsnorm.cu): argument rules shared with glu_api.cu.
constexpr int64_t kRmsMaxCols = 32768;
int validate_add_rmsnorm(const void *x, int64_t x_stride, const void *res, int64_t res_stride,
                         const void *gamma, const void *h, int64_t h_stride, const void *y, int64_t y_stride,
                         const float *rstd, int64_t n_rows, int64_t n_cols, float eps, int dtype, bool *empty);
constexpr int64_t kRmsBwdMaxCols = 16384;
int validate_add_rmsnorm_bwd(const void *dy, int64_t dy_stride, const void *h, int64_t h_stride, const float *rstd,
                             const void *gamma, const void *dh, int64_t dh_stride, const void *dx, int64_t dx_stride,
                             const void *dres, int64_t dres_stride, const float *dgamma, int64_t n_rows,
                             int64_t n_cols, int dtype, bool *empty);

// One validated call: what the planner needs.  Strides are in elements.
struct Call {
    int dir, act, dtype, E;
    int64_t rows, cols;
    const char *a, *b, *dc;
    char *y0, *y1;
    int64_t sa, sb, sdc, sy0, sy1;
    bool empty;   // n_rows == 0 or n_cols == 0: nothing to do
};

// Argument rules of glu_fwd / glu_bwd (include/glu.h), shared by the device
// and the host-memory entry points.  Pure host logic: no CUDA call.  On
// GLU_OK, *c describes the call with the [gate | up] layout resolved into
// separate operands.
int validate_fwd(const void *a, int64_t a_stride, const void *b, int64_t b_stride, const void *y,
                 int64_t y_stride, int64_t n_rows, int64_t n_cols, int layout, int act, int dtype,
                 Call *c);
int validate_bwd(const void *dc, int64_t dc_stride, const void *a, int64_t a_stride, const void *b,
                 int64_t b_stride, const void *da, int64_t da_stride, const void *db,
                 int64_t db_stride, int64_t n_rows, int64_t n_cols, int layout, int act, int dtype,
                 Call *c);

// Records the text of a CUDA error for glu_last_cuda_error() and returns GLU_ERR_CUDA.
int cuda_fail(cudaError_t e);

}  // namespace glu
