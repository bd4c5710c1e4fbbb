/*
 * glu.h - C ABI of the fused gated-activation library (GB300, sm_103a).
 *
 * The library computes the activation step of a gated MLP,
 *
 *     y = act(a) * b                                   (forward)
 *     da = dc * act'(a) * b,   db = dc * act(a)        (backward)
 *
 * element by element, where a is the gate projection's output, b the up
 * projection's output and dc the gradient arriving at y.  Sources:
 *   - "Skill: Write a Triton SiLU-Mul (SwiGLU) Kernel": Purpose (y = silu(a)*b
 *     between the gate/up and down projections; GeGLU and ReGLU on the same
 *     skeleton), Required reasoning process steps 1-9 (fp32 activation, cast at
 *     the store, the GeGLU erf form, the [gate | up] layout, the backward),
 *     Common failure modes (the tanh form of GELU, in-place over b, strides
 *     from tensor metadata).
 *   - "Kernel Profile: SwiGLU (Tier 1 - Element-wise)": Backward Pass
 *     (gradient formulas, sigmoid recomputed from a) and Key Patterns (in-place
 *     backward into a and b, no intermediate allocations).
 *
 * Conventions shared by every entry point
 *   - All pointers are DEVICE pointers into memory the caller owns.  The
 *     library allocates nothing, keeps no pointer after the call returns, and
 *     is asynchronous: work is enqueued on `stream` (NULL = the legacy default
 *     stream) and the call returns before it runs.  Pinned host memory
 *     (cudaHostAlloc, cudaHostRegister) is device memory in this sense: the
 *     kernels then read and write it in place over the host link (zero-copy),
 *     except the operands of the tensor-core entry points (glu_gemm_fwd,
 *     glu_gemm_nt, glu_mlp_fwd) and glu_add_rmsnorm_bwd's dgamma, which must
 *     be in device memory.
 *   - Matrices are row-major with a contiguous last dimension: element (r, c)
 *     of operand X is at X + r * X_stride + c.  Strides are in ELEMENTS of
 *     `dtype`, not bytes, and are ignored when n_rows == 1.
 *   - Every operand has the same dtype; outputs have the input dtype.  The
 *     activation runs in fp32 and the result is rounded to nearest-even once,
 *     at the store.  No flush-to-zero.
 *   - An output may be exactly the same matrix as an input (same pointer, same
 *     stride): each element's inputs are read before its outputs are written,
 *     and no two threads touch the same element.  Any other overlap between an
 *     output and an input, or any overlap between two outputs, is rejected
 *     with GLU_ERR_ALIAS.
 *   - Arguments are validated on the host before anything is launched; a
 *     negative return means nothing was enqueued.  n_rows == 0 or n_cols == 0
 *     returns GLU_OK without launching (pointers may then be NULL).
 *   - Pointers and strides that are 32- or 16-byte aligned use 256- or 128-bit
 *     memory accesses; any other alignment is valid and uses element-wide
 *     accesses.  Alignment is never an error, except for the operands that
 *     the tensor-core entry points read through the tensor-memory accelerator.
 *   - Non-finite inputs are outside the numerical contract; they do not fault.
 */
#ifndef GLU_H
#define GLU_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GLU_VERSION 1

/* Same type as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st *glu_stream_t;

/* Activation applied to the gate operand a (never to b).
 *   SILU       silu(x) = x * sigmoid(x)
 *              ("Skill: Write a Triton SiLU-Mul (SwiGLU) Kernel", step 5)
 *   GELU_ERF   0.5 * x * (1 + erf(x / sqrt 2))                          (step 7)
 *   GELU_TANH  0.5 * x * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3)))
 *              (Common failure modes, "GELU variant mismatch")
 *   RELU       max(x, 0); its derivative is taken as 0 at x == 0 (Purpose). */
typedef enum {
    GLU_ACT_SILU = 0,
    GLU_ACT_GELU_ERF = 1,
    GLU_ACT_GELU_TANH = 2,
    GLU_ACT_RELU = 3
} glu_act_t;

/* SPLIT:  a and b are separate n_rows x n_cols matrices.
 * CONCAT: one matrix x of n_rows x (2*n_cols) holds [gate | up] per row:
 *         a = x[:, :n_cols], b = x[:, n_cols:2*n_cols]
 *         ("Skill: Write a Triton SiLU-Mul (SwiGLU) Kernel", Inputs item 4 and
 *         Required reasoning step 8; the gate half comes first). */
typedef enum {
    GLU_LAYOUT_SPLIT = 0,
    GLU_LAYOUT_CONCAT = 1
} glu_layout_t;

typedef enum {
    GLU_F32 = 0,
    GLU_F16 = 1,
    GLU_BF16 = 2
} glu_dtype_t;

typedef enum {
    GLU_OK = 0,
    GLU_ERR_NULL = -1,    /* a required pointer is NULL (with n_rows, n_cols > 0) */
    GLU_ERR_SHAPE = -2,   /* negative size, or a size whose byte extent overflows */
    GLU_ERR_STRIDE = -3,  /* a stride smaller than its row width, or negative */
    GLU_ERR_ALIAS = -4,   /* outputs overlap inputs other than exactly, or each other */
    GLU_ERR_ENUM = -5,    /* unknown act, layout or dtype */
    GLU_ERR_CUDA = -6,    /* the CUDA runtime refused a launch or copy; see glu_last_cuda_error() */
    GLU_ERR_WORKSPACE = -7, /* host-memory entry points, glu_mlp_fwd: workspace NULL or too small for one row */
    GLU_ERR_VALUE = -8      /* an argument out of range: glu_add_rmsnorm_fwd's eps, or an
                               operand of a tensor-core entry point or glu_add_rmsnorm_bwd's
                               dgamma that is not in device memory */
} glu_status_t;

/*
 * Forward: y[r, c] = round(act(a[r, c]) * b[r, c]) for r < n_rows, c < n_cols.
 *
 *   a, a_stride   SPLIT: gate matrix.  CONCAT: the x matrix (width 2*n_cols,
 *                 a_stride >= 2*n_cols); the gate is its first half.
 *   b, b_stride   SPLIT: up matrix (b_stride >= n_cols).  CONCAT: ignored
 *                 (the up half is x + n_cols with x's stride); pass NULL, 0.
 *   y, y_stride   output, n_rows x n_cols, y_stride >= n_cols.  In place over
 *                 the up operand: y = b, y_stride = b_stride (SPLIT) or
 *                 y = x + n_cols, y_stride = a_stride (CONCAT).
 *   stream        CUDA stream the kernel is enqueued on.
 * Returns GLU_OK or a negative glu_status_t.
 */
int glu_fwd(const void *a, int64_t a_stride,
            const void *b, int64_t b_stride,
            void *y, int64_t y_stride,
            int64_t n_rows, int64_t n_cols,
            glu_layout_t layout, glu_act_t act, glu_dtype_t dtype,
            glu_stream_t stream);

/*
 * Backward ("Kernel Profile: SwiGLU", Backward Pass):
 *   da[r, c] = round(dc[r, c] * act'(a[r, c]) * b[r, c])
 *   db[r, c] = round(dc[r, c] * act(a[r, c]))
 * act and act' are recomputed in fp32 from a; nothing is saved by the forward.
 *
 *   dc, dc_stride incoming gradient, n_rows x n_cols.
 *   a, b          as in glu_fwd (CONCAT: a is x, b is ignored).
 *   da, da_stride SPLIT: gradient of a.  CONCAT: the dx matrix (width
 *                 2*n_cols, da_stride >= 2*n_cols); da fills its first half and
 *                 db its second.  In place ("Key Patterns", in-place backward):
 *                 da = a with da_stride = a_stride (CONCAT: dx = x).
 *   db, db_stride SPLIT: gradient of b; in place: db = b, db_stride = b_stride.
 *                 CONCAT: ignored (db is dx + n_cols); pass NULL, 0.
 * Returns GLU_OK or a negative glu_status_t.
 */
int glu_bwd(const void *dc, int64_t dc_stride,
            const void *a, int64_t a_stride,
            const void *b, int64_t b_stride,
            void *da, int64_t da_stride,
            void *db, int64_t db_stride,
            int64_t n_rows, int64_t n_cols,
            glu_layout_t layout, glu_act_t act, glu_dtype_t dtype,
            glu_stream_t stream);

/*
 * Host-memory variants.  Same computation, arguments and rules as glu_fwd /
 * glu_bwd (layouts, strides in elements, exact in-place aliasing, status
 * codes), except that every matrix argument is a HOST pointer.  Blocks of
 * rows are copied into `workspace`, processed by the same kernels, and copied
 * back; two workspace slots alternate so that the copy in of one block, the
 * kernel of the previous one and the copy out of the one before overlap.
 *
 *   workspace, workspace_bytes
 *                 DEVICE memory owned by the caller, at least
 *                 glu_host_workspace_bytes(1, ...) bytes (256-byte aligned is
 *                 best).  More workspace means larger blocks and fewer copies;
 *                 the library allocates nothing.  It must not be used by other
 *                 work until the call's work has completed.
 *   copy_in, compute, copy_out
 *                 streams for the host-to-device copies, the kernels and the
 *                 device-to-host copies.  They may be the same stream (no
 *                 overlap).  Work already enqueued on `compute` is finished
 *                 before the first copy; work enqueued on `compute` after the
 *                 call runs after the last copy out, so synchronising `compute`
 *                 is enough to see the outputs.
 * Host memory that is not page-locked is valid but its copies do not overlap.
 * On GLU_ERR_CUDA part of the work may have been enqueued and the outputs are
 * unspecified.
 */
int glu_fwd_host(const void *a, int64_t a_stride,
                 const void *b, int64_t b_stride,
                 void *y, int64_t y_stride,
                 int64_t n_rows, int64_t n_cols,
                 glu_layout_t layout, glu_act_t act, glu_dtype_t dtype,
                 void *workspace, size_t workspace_bytes,
                 glu_stream_t copy_in, glu_stream_t compute, glu_stream_t copy_out);

int glu_bwd_host(const void *dc, int64_t dc_stride,
                 const void *a, int64_t a_stride,
                 const void *b, int64_t b_stride,
                 void *da, int64_t da_stride,
                 void *db, int64_t db_stride,
                 int64_t n_rows, int64_t n_cols,
                 glu_layout_t layout, glu_act_t act, glu_dtype_t dtype,
                 void *workspace, size_t workspace_bytes,
                 glu_stream_t copy_in, glu_stream_t compute, glu_stream_t copy_out);

/*
 * glu_fwd_host without a caller workspace, for callers that cannot allocate
 * device memory at all: a plug-in inside an application whose own allocator
 * owns the device memory and gives none out, or a process that fixes its
 * memory budget at start-up and must not allocate while running.  The source
 * pages have no counterpart to this entry point; it is a deployment aid.
 *
 * Same arguments and rules as glu_fwd_host minus the workspace; one stream
 * carries the copies and the kernels, in order.  Blocks of rows are staged in
 * a fixed device array of GLU_NOALLOC_SCRATCH_BYTES inside the library, which
 * every GPU that loads the library holds until the process exits.  Nothing is
 * allocated: no cudaMalloc, no cudaFree, no event or stream creation.
 *   - A row that does not fit the array (inputs and output of one row, for
 *     SPLIT 3 * n_cols elements, for CONCAT 3 * n_cols) is rejected with
 *     GLU_ERR_WORKSPACE.
 *   - The first call on each device looks up the array's device address (a
 *     CUDA runtime query); make that first call before any stream capture.
 *     A device reset (cudaDeviceReset) reloads the library's module and may
 *     move the array: the address kept from before is then stale.  A call
 *     whose copy fails forgets it, so the next call looks it up again.
 *   - Every call uses the same array, which keeps the last call's contents
 *     (no part of it needs to start at zero): calls whose work can overlap on
 *     the GPU race on it, so order them, e.g. on one stream.
 */
#define GLU_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

int glu_fwd_host_noalloc(const void *a, int64_t a_stride,
                         const void *b, int64_t b_stride,
                         void *y, int64_t y_stride,
                         int64_t n_rows, int64_t n_cols,
                         glu_layout_t layout, glu_act_t act, glu_dtype_t dtype,
                         glu_stream_t stream);

/* Workspace bytes glu_fwd_host (backward == 0) or glu_bwd_host (backward != 0)
 * needs for blocks of `rows_per_block` rows of `n_cols` columns; 0 for invalid
 * arguments. */
size_t glu_host_workspace_bytes(int64_t rows_per_block, int64_t n_cols, glu_layout_t layout,
                                glu_dtype_t dtype, int backward);

/* Static English text for a glu_status_t value; never NULL. */
const char *glu_status_string(int status);

/* Text of the CUDA error behind this thread's most recent GLU_ERR_CUDA, or ""
 * if there was none.  Valid until the next call on the same thread. */
const char *glu_last_cuda_error(void);

/* GLU_VERSION of the loaded library. */
int glu_version(void);

/* What this thread's most recent successful glu_fwd / glu_bwd / glu_gemm_fwd
 * enqueued.  `launched` is 0 when the call was a no-op (an empty matrix).
 * For glu_gemm_fwd: path = 3, unroll = blocks per cluster (1, or 2 for a pair
 * sharing each tile), vec_bytes = bytes per row of
 * each y store (64: 32 x 32 boxes through the tensor-memory accelerator, used
 * when y, its row stride and its row width are 16-byte multiples; else 16 or
 * 2 from registers), grid =
 * blocks of the persistent grid, vector_units = tiles of y, and threads as
 * launched; the other fields are 0.  For glu_add_rmsnorm_fwd and
 * glu_add_rmsnorm_bwd: vector_units = rows, unroll = elements per thread and
 * row, vec_bytes 16 or the element size, and path names the kernel: 4 the
 * forward, or the backward with element accesses; the backward on 16-byte
 * rows 6 (rows staged in shared memory), 7 (narrow rows held in registers,
 * one block per group of rows) or 8 (persistent teams of registers). */
typedef struct {
    int32_t launched;     /* 1 if a kernel was enqueued */
    int32_t backward;     /* 0 = forward kernel, 1 = backward kernel */
    int32_t vec_bytes;    /* bytes per operand per memory access: 32, 16 or the element size */
    int32_t unroll;       /* accesses each thread keeps in flight per operand */
    int32_t threads;      /* threads per block */
    int32_t grid;         /* blocks launched */
    int32_t flattened;    /* 1 if the rows were contiguous and walked as one row */
    int32_t path;         /* 1 = direct loads, 2 = bulk copies staged in shared memory, 3 = GEMM */
    int64_t vector_units; /* full-width accesses per operand */
    int64_t tail_elems;   /* elements handled one at a time (row ends) */
} glu_launch_info_t;

/* Copies this thread's last launch description into *out.  GLU_ERR_NULL if out is NULL. */
int glu_last_launch(glu_launch_info_t *out);

/* Process-wide launch tuning (used by benchmarks and tuning sweeps; the
 * defaults are what the library was tuned to).  A field left at 0 means
 * "library default".  Not synchronised with concurrent glu_fwd/glu_bwd calls
 * on other threads.
 *   vec_bytes     upper bound on the access width: 32, 16, or the element size
 *   unroll        1, 2 or 4 accesses in flight per operand per thread
 *   ctas_per_sm   >0: persistent grid of that many blocks per SM;
 *                 <0: one block per tile of work (no grid-stride reuse)
 *   dependent_launch
 *                 0 or 1: launch with a programmatic dependency on the previous
 *                 kernel in the stream (the kernel still waits for that grid to
 *                 finish before touching memory, so results and ordering are
 *                 unchanged; only scheduling overlaps); -1: ordinary launch
 *   path          0 or 1: direct 16/32-byte loads into registers; 2: for
 *                 contiguous, 16-byte aligned operands whose inputs are in
 *                 device memory, whole 16 KiB chunks are staged in shared
 *                 memory by the bulk-copy engine (one block per SM) and the
 *                 rest takes the direct path; everything else takes it too */
typedef struct {
    int32_t vec_bytes;
    int32_t unroll;
    int32_t ctas_per_sm;
    int32_t dependent_launch;
    int32_t path;
} glu_tuning_t;

int glu_set_tuning(const glu_tuning_t *t);   /* GLU_ERR_ENUM for unsupported values */
int glu_get_tuning(glu_tuning_t *out);

/* Kernels that wait on the bulk-copy engine or the tensor cores (the bulk-copy
 * path, glu_gemm_fwd and glu_add_rmsnorm_bwd's staged kernel) bound every wait
 * (about a second) and count the waits that ran out on the current device
 * instead of hanging.
 * Copies that count into *count (synchronising with the device) and, if
 * `reset`, sets it back to 0.  A nonzero count means some outputs of those
 * launches were not written. */
int glu_wait_timeouts(unsigned int *count, int reset);

/* Self-test of that bound: enqueues on `stream` one warp that waits on a
 * shared-memory barrier nothing arrives on, with the same bounded wait.  The
 * wait runs out after about a second, the kernel returns, and the count of
 * glu_wait_timeouts() goes up by one; the context stays usable.  Returns
 * GLU_OK, or GLU_ERR_CUDA if the launch is refused. */
int glu_wait_selftest(glu_stream_t stream);

/*
 * Gate and up projections with the gated activation applied in the GEMM
 * epilogue, on the tensor cores:
 *
 *     y[m, i] = round(act(g[m, i]) * u[m, i]),
 *     g[m, i] = sum_k x[m, k] * w_gate[i, k],   u[m, i] = sum_k x[m, k] * w_up[i, k].
 *
 * Sources: "Skill: Write a Triton SiLU-Mul (SwiGLU) Kernel" (Purpose; "Versus
 * epilogue fusion" under Performance requirements: the gate and up tiles stay
 * on chip and only y reaches HBM) and "Fused Kernels" (section 4, "The fused
 * MLP": gate and up tiles as x @ gate^T and x @ up^T, the activation applied
 * to them in registers).  g and u are accumulated in fp32 (products of
 * 16-bit values are exact in fp32; the order of the additions is the
 * hardware's), then the activation runs in fp32 as in glu_fwd and the result
 * is rounded to nearest-even once.
 *
 *   x, x_stride        M x K activations (row-major, element stride x_stride >= K).
 *   w_gate, w_up       I x K weights, row i holding output feature i (the
 *                      nn.Linear layout), both with row stride w_stride >= K.
 *   y, y_stride        M x I output, y_stride >= I.  y must not overlap x or
 *                      the weights (GLU_ERR_ALIAS).
 *   act                any glu_act_t.
 *   dtype              GLU_F16 or GLU_BF16 (the tensor cores take both operands
 *                      in one 16-bit type); GLU_F32 returns GLU_ERR_ENUM.
 *   stream             CUDA stream the kernel is enqueued on.
 * The operands are read by the tensor-memory accelerator: x, w_gate and w_up
 * must be 16-byte aligned and x_stride, w_stride multiples of 8 elements,
 * else GLU_ERR_STRIDE (y has no alignment rule).  M, K, I < 2^31.  M == 0 or
 * I == 0 returns GLU_OK without work; K == 0 sets y to 0 (act(0) * 0).
 * All pointers must be device memory (cudaMalloc and the like; checked with
 * cudaPointerGetAttributes, else GLU_ERR_VALUE); the library keeps none after
 * the call.  A wait that runs out of its time budget (about a second) is counted for
 * glu_wait_timeouts() and leaves that block's outputs unwritten.
 * Returns GLU_OK or a negative glu_status_t.
 */
int glu_gemm_fwd(const void *x, int64_t x_stride,
                 const void *w_gate, const void *w_up, int64_t w_stride,
                 void *y, int64_t y_stride,
                 int64_t M, int64_t K, int64_t I,
                 glu_act_t act, glu_dtype_t dtype, glu_stream_t stream);

/*
 * The plain product on the same tensor-core kernel, the down projection of
 * the MLP ("Fused Kernels", section 4, "The fused MLP": the gated tile times
 * the down weights; "Skill: Write a Triton SiLU-Mul (SwiGLU) Kernel",
 * Purpose: down_proj of the gated product):
 *
 *     d[m, n] = round(sum_k a[m, k] * b[n, k]),
 *
 * sums in fp32 in the hardware's order, one rounding to nearest-even.
 *   a, a_stride        M x K (row-major, a_stride >= K).
 *   b, b_stride        N x K, row n holding output feature n (the nn.Linear
 *                      layout), b_stride >= K.
 *   d, d_stride        M x N output, d_stride >= N; no overlap with a or b
 *                      (GLU_ERR_ALIAS).
 *   dtype              GLU_F16 or GLU_BF16.
 * Alignment, device-memory, empty-size, K == 0 (d = 0) and timeout rules as
 * glu_gemm_fwd.  glu_last_launch reports path = 5.
 */
int glu_gemm_nt(const void *a, int64_t a_stride,
                const void *b, int64_t b_stride,
                void *d, int64_t d_stride,
                int64_t M, int64_t K, int64_t N,
                glu_dtype_t dtype, glu_stream_t stream);

/*
 * The gated MLP, out = down_proj(act(gate_proj(x)) * up_proj(x)) ("Skill:
 * Write a Triton SiLU-Mul (SwiGLU) Kernel", Purpose; "Fused Kernels", section
 * 4, "The fused MLP"):
 *
 *     y[m, i]   = round(act(x[m] . w_gate[i]) * (x[m] . w_up[i]))   (glu_gemm_fwd)
 *     out[m, h] = round(y[m] . w_down[h])                           (glu_gemm_nt)
 *
 * y, rounded once to the dtype as glu_gemm_fwd stores it, goes through the
 * caller's workspace: the rows run in chunks whose y fits it (at most 1 GiB
 * of y per chunk), two launches per chunk.  Keeping y in registers or tensor
 * memory instead, as the page's kernel does, would recompute the gate and up
 * products once per output column tile (16 times at H = 4096); chunks small
 * enough for y to stay in L2 between the products were measured slower on
 * GB300 than whole-batch launches (0.847 against 0.778 ms at 4096 x 4096 x
 * 14336 bf16): smaller launches lose more to tile rounds than the y traffic
 * costs.
 *   x, x_stride        M x H activations, x_stride >= H.
 *   w_gate, w_up       I x H, row stride w_stride >= H.
 *   w_down             H x I (row h holds output feature h), w_down_stride >= I.
 *   out, out_stride    M x H output, out_stride >= H; no overlap with any
 *                      operand or the workspace (GLU_ERR_ALIAS).
 *   workspace          device memory for one chunk's y, 16-byte aligned:
 *                      glu_mlp_workspace_bytes(M, I, dtype) bytes, or less
 *                      (smaller chunks), but at least one row of
 *                      round_up(I, 8) elements, else GLU_ERR_WORKSPACE.  It
 *                      holds the last chunk's y on return.
 * x, the weights, the workspace and out must be device memory (GLU_ERR_VALUE)
 * with 16-byte aligned bases and strides that are multiples of 8 elements
 * (GLU_ERR_STRIDE); both are checked before the first launch.  M == 0 or
 * H == 0: no work; I == 0: out = 0.  Two launches per chunk on `stream`;
 * glu_last_launch describes the last.  Returns GLU_OK or a negative
 * glu_status_t.
 */
int glu_mlp_fwd(const void *x, int64_t x_stride,
                const void *w_gate, const void *w_up, int64_t w_stride,
                const void *w_down, int64_t w_down_stride,
                void *out, int64_t out_stride,
                int64_t M, int64_t H, int64_t I,
                glu_act_t act, glu_dtype_t dtype,
                void *workspace, size_t workspace_bytes, glu_stream_t stream);

/* Workspace bytes for glu_mlp_fwd to run M rows of intermediate size I in
 * one chunk (the y of all rows, rows of round_up(I, 8) elements), capped at
 * 1 GiB (chunks of whole 256-row blocks); 0 for invalid arguments. */
size_t glu_mlp_workspace_bytes(int64_t M, int64_t I, glu_dtype_t dtype);

/*
 * Fused residual add + RMSNorm ("Skill: Write a Triton Fused Add+RMSNorm
 * Kernel": Purpose; Required reasoning process steps 1-9; Kernel design rules;
 * Correctness requirements), over each row r < n_rows of H = n_cols elements:
 *
 *     s[r, j] = x[r, j] + residual[r, j]             (fp32; exact for 16-bit inputs)
 *     h[r, j] = round(s[r, j])                        (the residual stream for the next block)
 *     rstd[r] = 1 / sqrt(sum_j s[r, j]^2 / H + eps)   (eps inside the root)
 *     y[r, j] = round(s[r, j] * rstd[r] * gamma[j])   (gamma indexed by column only)
 *
 * No mean is subtracted and there is no bias.  Arithmetic is fp32 from the add
 * through the product; each stored value is rounded to nearest-even once.
 *
 *   x, x_stride          input rows (row-major, element strides, >= n_cols).
 *   residual, res_stride the residual rows.
 *   gamma                n_cols elements of `dtype`, shared by every row.
 *   h, h_stride          output: the summed rows.  May be exactly x or exactly
 *                        residual (same pointer and stride): in place.
 *   y, y_stride          output: the normalised rows.  May be exactly x or
 *                        residual when h is not the same one; h and y must not
 *                        overlap.  Other overlaps with an input: GLU_ERR_ALIAS.
 *   rstd                 NULL, or n_rows floats receiving rstd (kept for a
 *                        backward pass); must not overlap any matrix.
 *   eps                  > 0 and finite, else GLU_ERR_VALUE.
 *   n_cols               at most 32768 (a row lives in registers), else
 *                        GLU_ERR_SHAPE.
 * All pointers are device pointers; the call is asynchronous on `stream`.
 * n_rows == 0 or n_cols == 0 returns GLU_OK without launching.
 * Returns GLU_OK or a negative glu_status_t.
 */
int glu_add_rmsnorm_fwd(const void *x, int64_t x_stride,
                        const void *residual, int64_t res_stride,
                        const void *gamma,
                        void *h, int64_t h_stride,
                        void *y, int64_t y_stride,
                        float *rstd,
                        int64_t n_rows, int64_t n_cols, float eps,
                        glu_dtype_t dtype, glu_stream_t stream);

/*
 * Backward of glu_add_rmsnorm_fwd ("Skill: Write a Triton Fused Add+RMSNorm
 * Kernel", Required reasoning process steps 9-10: the forward keeps rstd and
 * the summed rows h; the gradient of the norm goes to x and to the residual
 * alike).  For each row, with s = h (the stored sum) and rstd as the forward
 * kept it:
 *
 *     ds[j]     = rstd * gamma[j] * dy[j] - (rstd^3 / H) * s[j] * sum_k gamma[k] dy[k] s[k]
 *                 (+ dh[j], the gradient reaching h through the residual stream)
 *     dx[j]     = round(ds[j])            (the gradient of x and of the residual)
 *     dgamma[j] += sum over rows of dy[j] * s[j] * rstd
 *
 * in fp32 (the row sum with fused multiply-adds, reduced over the block).
 *
 *   dy, dy_stride        gradient arriving at y.
 *   h, h_stride          the sums the forward stored.
 *   rstd                 n_rows floats from the forward.
 *   gamma                n_cols elements of `dtype`.
 *   dh, dh_stride        NULL, or the gradient arriving at h.
 *   dx, dx_stride        output.  May be exactly dy, h or dh (in place).
 *   dres, dres_stride    NULL, or a second output receiving the same values
 *                        (the residual's gradient); may be exactly one of the
 *                        inputs that dx is not.  dx and dres must not overlap.
 *   dgamma               NULL, or n_cols floats that the row sums are ADDED to
 *                        (zero it for a fresh gradient).  The additions from
 *                        different blocks arrive in no fixed order.  It must
 *                        be in device memory (it takes atomic reductions),
 *                        else GLU_ERR_VALUE.
 *   n_cols               at most 16384, else GLU_ERR_SHAPE.
 * Other rules as glu_add_rmsnorm_fwd (device pointers, element strides,
 * GLU_ERR_ALIAS for any other overlap, asynchronous on `stream`).
 *
 * Rows whose operands are 16-byte aligned (bases, strides, width) and whose
 * inputs dy, h, dh and rstd are in device memory use 16-byte accesses: rows of
 * up to 512 16-byte vectors (384 for f32) are loaded straight into registers (narrow rows,
 * up to 128 vectors, one block per group of rows when the launch fits on the
 * GPU at once; otherwise a persistent grid of teams of threads, one row per
 * team at a time), wider rows are staged in shared memory by the bulk-copy
 * engine.  Every wait of the staged kernel is bounded (about a second); one
 * that runs out is counted by glu_wait_timeouts() and leaves that launch's
 * outputs and dgamma incomplete.  Other rows (pinned host inputs included)
 * use element accesses.
 */
int glu_add_rmsnorm_bwd(const void *dy, int64_t dy_stride,
                        const void *h, int64_t h_stride,
                        const float *rstd,
                        const void *gamma,
                        const void *dh, int64_t dh_stride,
                        void *dx, int64_t dx_stride,
                        void *dres, int64_t dres_stride,
                        float *dgamma,
                        int64_t n_rows, int64_t n_cols,
                        glu_dtype_t dtype, glu_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GLU_H */
