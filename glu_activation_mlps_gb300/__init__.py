"""Python binding of the fused gated-activation library (GB300, sm_103a).

``libglu_gb300.so`` exports the C ABI declared in ``include/glu.h``.  This
module only marshals arguments: every step of the computation runs in the
library's CUDA kernels.  There is no CPU fallback; if the library has not been
built, every call raises.

Two levels:
  * ``glu_fwd`` / ``glu_bwd`` / ``glu_status_string`` / ... : the C entry points
    with the same names and arguments (raw device addresses as ints, strides
    in elements, enum codes, the stream handle as an int);
  * ``fwd`` / ``bwd``: the same calls taking torch CUDA tensors, reading
    pointers and strides from the tensors' metadata.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libglu_gb300.so")

ACT = {"silu": 0, "gelu_erf": 1, "gelu_tanh": 2, "relu": 3}
LAYOUT = {"split": 0, "concat": 1}
DTYPE = {"f32": 0, "f16": 1, "bf16": 2}
STATUS = {0: "GLU_OK", -1: "GLU_ERR_NULL", -2: "GLU_ERR_SHAPE", -3: "GLU_ERR_STRIDE",
          -4: "GLU_ERR_ALIAS", -5: "GLU_ERR_ENUM", -6: "GLU_ERR_CUDA", -7: "GLU_ERR_WORKSPACE",
          -8: "GLU_ERR_VALUE"}

# Every symbol include/glu.h declares.
EXPORTS = ("glu_fwd", "glu_bwd", "glu_fwd_host", "glu_bwd_host", "glu_fwd_host_noalloc",
           "glu_host_workspace_bytes",
           "glu_status_string", "glu_last_cuda_error", "glu_version", "glu_last_launch",
           "glu_set_tuning", "glu_get_tuning", "glu_wait_timeouts", "glu_wait_selftest", "glu_gemm_fwd",
           "glu_gemm_nt", "glu_mlp_fwd", "glu_mlp_workspace_bytes",
           "glu_add_rmsnorm_fwd", "glu_add_rmsnorm_bwd")


class GluError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {STATUS.get(status, status)} ({glu_status_string(status)})"
        if status == -6:
            msg += ": " + glu_last_cuda_error()
        super().__init__(msg)


class LaunchInfo(ctypes.Structure):
    _fields_ = [("launched", ctypes.c_int32), ("backward", ctypes.c_int32),
                ("vec_bytes", ctypes.c_int32), ("unroll", ctypes.c_int32),
                ("threads", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("flattened", ctypes.c_int32), ("path", ctypes.c_int32),
                ("vector_units", ctypes.c_int64), ("tail_elems", ctypes.c_int64)]


class Tuning(ctypes.Structure):
    _fields_ = [("vec_bytes", ctypes.c_int32), ("unroll", ctypes.c_int32),
                ("ctas_per_sm", ctypes.c_int32), ("dependent_launch", ctypes.c_int32),
                ("path", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    from . import _build
    return _build.build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(glu_activation_mlps_gb300.build()); there is no CPU fallback")
            L = ctypes.CDLL(LIB_PATH)
            i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
            L.glu_fwd.argtypes = [vp, i64, vp, i64, vp, i64, i64, i64, ci, ci, ci, vp]
            L.glu_fwd.restype = ci
            L.glu_bwd.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, i64, i64, ci, ci, ci, vp]
            L.glu_bwd.restype = ci
            sz = ctypes.c_size_t
            L.glu_fwd_host.argtypes = [vp, i64, vp, i64, vp, i64, i64, i64, ci, ci, ci, vp, sz, vp, vp, vp]
            L.glu_fwd_host.restype = ci
            L.glu_bwd_host.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, i64, i64, ci, ci, ci,
                                       vp, sz, vp, vp, vp]
            L.glu_bwd_host.restype = ci
            L.glu_fwd_host_noalloc.argtypes = [vp, i64, vp, i64, vp, i64, i64, i64, ci, ci, ci, vp]
            L.glu_fwd_host_noalloc.restype = ci
            L.glu_host_workspace_bytes.argtypes = [i64, i64, ci, ci, ci]
            L.glu_host_workspace_bytes.restype = sz
            L.glu_status_string.argtypes = [ci]
            L.glu_status_string.restype = ctypes.c_char_p
            L.glu_last_cuda_error.argtypes = []
            L.glu_last_cuda_error.restype = ctypes.c_char_p
            L.glu_version.argtypes = []
            L.glu_version.restype = ci
            L.glu_last_launch.argtypes = [ctypes.POINTER(LaunchInfo)]
            L.glu_last_launch.restype = ci
            L.glu_set_tuning.argtypes = [ctypes.POINTER(Tuning)]
            L.glu_set_tuning.restype = ci
            L.glu_get_tuning.argtypes = [ctypes.POINTER(Tuning)]
            L.glu_get_tuning.restype = ci
            L.glu_wait_timeouts.argtypes = [ctypes.POINTER(ctypes.c_uint), ci]
            L.glu_wait_timeouts.restype = ci
            L.glu_wait_selftest.argtypes = [vp]
            L.glu_wait_selftest.restype = ci
            L.glu_gemm_fwd.argtypes = [vp, i64, vp, vp, i64, vp, i64, i64, i64, i64, ci, ci, vp]
            L.glu_gemm_fwd.restype = ci
            L.glu_gemm_nt.argtypes = [vp, i64, vp, i64, vp, i64, i64, i64, i64, ci, vp]
            L.glu_gemm_nt.restype = ci
            L.glu_mlp_fwd.argtypes = [vp, i64, vp, vp, i64, vp, i64, vp, i64, i64, i64, i64, ci, ci, vp, sz, vp]
            L.glu_mlp_fwd.restype = ci
            L.glu_mlp_workspace_bytes.argtypes = [i64, i64, ci]
            L.glu_mlp_workspace_bytes.restype = sz
            L.glu_add_rmsnorm_fwd.argtypes = [vp, i64, vp, i64, vp, vp, i64, vp, i64, vp, i64, i64,
                                              ctypes.c_float, ci, vp]
            L.glu_add_rmsnorm_fwd.restype = ci
            L.glu_add_rmsnorm_bwd.argtypes = [vp, i64, vp, i64, vp, vp, vp, i64, vp, i64, vp, i64, vp, i64, i64,
                                              ci, vp]
            L.glu_add_rmsnorm_bwd.restype = ci
            _lib = L
    return _lib


# ---- the C entry points -------------------------------------------------------

def glu_fwd(a, a_stride, b, b_stride, y, y_stride, n_rows, n_cols, layout, act, dtype, stream) -> int:
    return lib().glu_fwd(a, a_stride, b, b_stride, y, y_stride, n_rows, n_cols,
                         layout, act, dtype, stream)


def glu_bwd(dc, dc_stride, a, a_stride, b, b_stride, da, da_stride, db, db_stride,
            n_rows, n_cols, layout, act, dtype, stream) -> int:
    return lib().glu_bwd(dc, dc_stride, a, a_stride, b, b_stride, da, da_stride, db, db_stride,
                         n_rows, n_cols, layout, act, dtype, stream)


def glu_fwd_host(a, a_stride, b, b_stride, y, y_stride, n_rows, n_cols, layout, act, dtype,
                 workspace, workspace_bytes, copy_in, compute, copy_out) -> int:
    return lib().glu_fwd_host(a, a_stride, b, b_stride, y, y_stride, n_rows, n_cols, layout, act, dtype,
                              workspace, workspace_bytes, copy_in, compute, copy_out)


def glu_bwd_host(dc, dc_stride, a, a_stride, b, b_stride, da, da_stride, db, db_stride, n_rows, n_cols,
                 layout, act, dtype, workspace, workspace_bytes, copy_in, compute, copy_out) -> int:
    return lib().glu_bwd_host(dc, dc_stride, a, a_stride, b, b_stride, da, da_stride, db, db_stride,
                              n_rows, n_cols, layout, act, dtype, workspace, workspace_bytes,
                              copy_in, compute, copy_out)


def glu_fwd_host_noalloc(a, a_stride, b, b_stride, y, y_stride, n_rows, n_cols, layout, act, dtype,
                         stream) -> int:
    """glu_fwd_host staged through the library's own fixed device array: for
    callers that cannot allocate device memory (see include/glu.h)."""
    return lib().glu_fwd_host_noalloc(a, a_stride, b, b_stride, y, y_stride, n_rows, n_cols, layout,
                                      act, dtype, stream)


def glu_host_workspace_bytes(rows_per_block, n_cols, layout, dtype, backward) -> int:
    return lib().glu_host_workspace_bytes(rows_per_block, n_cols, layout, dtype, backward)


def glu_status_string(status: int) -> str:
    return lib().glu_status_string(status).decode()


def glu_last_cuda_error() -> str:
    return lib().glu_last_cuda_error().decode()


def glu_version() -> int:
    return lib().glu_version()


def glu_last_launch() -> dict:
    info = LaunchInfo()
    st = lib().glu_last_launch(ctypes.byref(info))
    if st:
        raise GluError(st, "glu_last_launch")
    return {f: getattr(info, f) for f, _ in LaunchInfo._fields_}


def glu_set_tuning(vec_bytes: int = 0, unroll: int = 0, ctas_per_sm: int = 0,
                   dependent_launch: int = 0, path: int = 0) -> None:
    t = Tuning(vec_bytes, unroll, ctas_per_sm, dependent_launch, path)
    st = lib().glu_set_tuning(ctypes.byref(t))
    if st:
        raise GluError(st, "glu_set_tuning")


def glu_wait_timeouts(reset: bool = False) -> int:
    c = ctypes.c_uint(0)
    st = lib().glu_wait_timeouts(ctypes.byref(c), int(reset))
    if st:
        raise GluError(st, "glu_wait_timeouts")
    return c.value


def glu_wait_selftest(stream=None) -> None:
    """Enqueue the bounded-wait self-test (one warp whose wait nothing
    completes; it returns after about a second and counts one timeout)."""
    st = lib().glu_wait_selftest(_stream(stream))
    if st:
        raise GluError(st, "glu_wait_selftest")


def glu_gemm_fwd(x, x_stride, w_gate, w_up, w_stride, y, y_stride, M, K, I, act, dtype, stream) -> int:
    return lib().glu_gemm_fwd(x, x_stride, w_gate, w_up, w_stride, y, y_stride, M, K, I, act, dtype, stream)


def glu_gemm_nt(a, a_stride, b, b_stride, d, d_stride, M, K, N, dtype, stream) -> int:
    return lib().glu_gemm_nt(a, a_stride, b, b_stride, d, d_stride, M, K, N, dtype, stream)


def glu_mlp_fwd(x, x_stride, w_gate, w_up, w_stride, w_down, w_down_stride, out, out_stride, M, H, I, act, dtype,
                workspace, workspace_bytes, stream) -> int:
    return lib().glu_mlp_fwd(x, x_stride, w_gate, w_up, w_stride, w_down, w_down_stride, out, out_stride, M, H, I,
                             act, dtype, workspace, workspace_bytes, stream)


def glu_mlp_workspace_bytes(M, I, dtype) -> int:
    return lib().glu_mlp_workspace_bytes(M, I, dtype)


def glu_add_rmsnorm_fwd(x, x_stride, residual, res_stride, gamma, h, h_stride, y, y_stride, rstd,
                        n_rows, n_cols, eps, dtype, stream) -> int:
    return lib().glu_add_rmsnorm_fwd(x, x_stride, residual, res_stride, gamma, h, h_stride, y, y_stride, rstd,
                                     n_rows, n_cols, eps, dtype, stream)


def glu_add_rmsnorm_bwd(dy, dy_stride, h, h_stride, rstd, gamma, dh, dh_stride, dx, dx_stride, dres, dres_stride,
                        dgamma, n_rows, n_cols, dtype, stream) -> int:
    return lib().glu_add_rmsnorm_bwd(dy, dy_stride, h, h_stride, rstd, gamma, dh, dh_stride, dx, dx_stride, dres,
                                     dres_stride, dgamma, n_rows, n_cols, dtype, stream)


def glu_get_tuning() -> dict:
    t = Tuning()
    st = lib().glu_get_tuning(ctypes.byref(t))
    if st:
        raise GluError(st, "glu_get_tuning")
    return {"vec_bytes": t.vec_bytes, "unroll": t.unroll, "ctas_per_sm": t.ctas_per_sm,
            "dependent_launch": t.dependent_launch, "path": t.path}


# ---- torch tensor marshalling -------------------------------------------------

def _dtype_code(t) -> int:
    import torch
    m = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
    if t.dtype not in m:
        raise TypeError(f"unsupported dtype {t.dtype}; expected float32, float16 or bfloat16")
    return m[t.dtype]


def _rows(t, name):
    """(n_rows, row stride) of a tensor viewed as a matrix over its last dim."""
    if t.dim() < 1 or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor with at least one dimension")
    if t.stride(-1) != 1 and t.shape[-1] > 1:
        raise ValueError(f"{name}: the last dimension must be contiguous")
    if t.dim() == 1:
        return 1, t.shape[0]
    lead = t.shape[:-1]
    # leading dims must collapse to one row index with a single stride
    stride = t.stride(-2)
    expect = stride
    for d in range(t.dim() - 2, -1, -1):
        if t.shape[d] != 1 and t.stride(d) != expect:
            raise ValueError(f"{name}: leading dimensions do not collapse to one row stride")
        expect *= t.shape[d]
    n = 1
    for s in lead:
        n *= s
    return n, stride


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def fwd(a, b=None, *, y=None, act: str = "silu", layout: str = "split", stream=None):
    """y = act(a) * b on CUDA tensors.  SPLIT: a, b of one shape (..., I).
    CONCAT: a is x of shape (..., 2I), b is None.  ``y`` may be given (also as
    b, or as x[..., I:], for in-place); otherwise it is allocated."""
    import torch
    if layout not in LAYOUT:
        raise ValueError(layout)
    concat = layout == "concat"
    n_rows, a_stride = _rows(a, "a")
    if concat:
        if a.shape[-1] % 2:
            raise ValueError("concat input needs an even last dimension")
        n_cols = a.shape[-1] // 2
        b_ptr, b_stride = None, 0
        out_shape = (*a.shape[:-1], n_cols)
    else:
        if b is None or b.shape != a.shape or b.dtype != a.dtype:
            raise ValueError("b must match a in shape and dtype")
        n_cols = a.shape[-1]
        _, b_stride = _rows(b, "b")
        b_ptr = b.data_ptr()
        out_shape = a.shape
    if y is None:
        y = torch.empty(out_shape, dtype=a.dtype, device=a.device)
    if tuple(y.shape) != tuple(out_shape) or y.dtype != a.dtype:
        raise ValueError("y has the wrong shape or dtype")
    _, y_stride = _rows(y, "y")
    st = glu_fwd(a.data_ptr(), a_stride, b_ptr, b_stride, y.data_ptr(), y_stride,
                 n_rows, n_cols, LAYOUT[layout], ACT[act], _dtype_code(a), _stream(stream))
    if st:
        raise GluError(st, "glu_fwd")
    return y


def bwd(dc, a, b=None, *, da=None, db=None, act: str = "silu", layout: str = "split",
        inplace: bool = False, stream=None):
    """(da, db) = (dc * act'(a) * b, dc * act(a)).  SPLIT returns (da, db);
    CONCAT (a = x, b None) returns dx = [da | db].  ``inplace`` writes da over
    a and db over b (dx over x)."""
    import torch
    concat = layout == "concat"
    n_rows, a_stride = _rows(a, "a")
    _, dc_stride = _rows(dc, "dc")
    code = _dtype_code(a)
    if concat:
        n_cols = a.shape[-1] // 2
        if dc.shape[-1] != n_cols:
            raise ValueError("dc must have half the width of x")
        dx = a if inplace else (da if da is not None else torch.empty_like(a))
        _, dx_stride = _rows(dx, "dx")
        st = glu_bwd(dc.data_ptr(), dc_stride, a.data_ptr(), a_stride, None, 0,
                     dx.data_ptr(), dx_stride, None, 0, n_rows, n_cols,
                     LAYOUT[layout], ACT[act], code, _stream(stream))
        if st:
            raise GluError(st, "glu_bwd")
        return dx
    if b is None or b.shape != a.shape or dc.shape != a.shape:
        raise ValueError("dc, a and b must have one shape")
    n_cols = a.shape[-1]
    _, b_stride = _rows(b, "b")
    if inplace:
        da, db = a, b
    da = da if da is not None else torch.empty_like(a)
    db = db if db is not None else torch.empty_like(b)
    _, da_stride = _rows(da, "da")
    _, db_stride = _rows(db, "db")
    st = glu_bwd(dc.data_ptr(), dc_stride, a.data_ptr(), a_stride, b.data_ptr(), b_stride,
                 da.data_ptr(), da_stride, db.data_ptr(), db_stride, n_rows, n_cols,
                 LAYOUT[layout], ACT[act], code, _stream(stream))
    if st:
        raise GluError(st, "glu_bwd")
    return da, db


def gemm_fwd(x, w_gate, w_up, *, y=None, act: str = "silu", stream=None):
    """y = act(x @ w_gate^T) * (x @ w_up^T) on the tensor cores, the activation
    applied in the GEMM epilogue.  x is (..., K); the weights are (I, K) in the
    nn.Linear layout and share one row stride; f16 or bf16."""
    import torch
    n_rows, x_stride = _rows(x, "x")
    if w_gate.dim() != 2 or w_up.shape != w_gate.shape or w_gate.shape[1] != x.shape[-1]:
        raise ValueError("w_gate and w_up must both be (I, K) with K = x.shape[-1]")
    if w_gate.dtype != x.dtype or w_up.dtype != x.dtype:
        raise ValueError("x and the weights must have one dtype")
    _, wg_stride = _rows(w_gate, "w_gate")
    _, wu_stride = _rows(w_up, "w_up")
    if wg_stride != wu_stride:
        raise ValueError("w_gate and w_up must have one row stride")
    n_out, K = w_gate.shape
    if y is None:
        y = torch.empty((*x.shape[:-1], n_out), dtype=x.dtype, device=x.device)
    if tuple(y.shape) != (*x.shape[:-1], n_out) or y.dtype != x.dtype:
        raise ValueError("y has the wrong shape or dtype")
    _, y_stride = _rows(y, "y")
    st = glu_gemm_fwd(x.data_ptr(), x_stride, w_gate.data_ptr(), w_up.data_ptr(), wg_stride,
                      y.data_ptr(), y_stride, n_rows, K, n_out, ACT[act], _dtype_code(x), _stream(stream))
    if st:
        raise GluError(st, "glu_gemm_fwd")
    return y


def gemm_nt(a, b, *, d=None, stream=None):
    """d = a @ b^T on the tensor cores (the MLP's down projection).  a is
    (..., K); b is (N, K) in the nn.Linear layout; f16 or bf16."""
    import torch
    n_rows, a_stride = _rows(a, "a")
    if b.dim() != 2 or b.shape[1] != a.shape[-1] or b.dtype != a.dtype:
        raise ValueError("b must be (N, K) with K = a.shape[-1] and a's dtype")
    _, b_stride = _rows(b, "b")
    N, K = b.shape
    if d is None:
        d = torch.empty((*a.shape[:-1], N), dtype=a.dtype, device=a.device)
    if tuple(d.shape) != (*a.shape[:-1], N) or d.dtype != a.dtype:
        raise ValueError("d has the wrong shape or dtype")
    _, d_stride = _rows(d, "d")
    st = glu_gemm_nt(a.data_ptr(), a_stride, b.data_ptr(), b_stride, d.data_ptr(), d_stride, n_rows, K, N,
                     _dtype_code(a), _stream(stream))
    if st:
        raise GluError(st, "glu_gemm_nt")
    return d


def mlp_fwd(x, w_gate, w_up, w_down, *, out=None, act: str = "silu", workspace=None, stream=None):
    """out = (act(x @ w_gate^T) * (x @ w_up^T)) @ w_down^T; x is (..., H), the
    gate and up weights (I, H), the down weights (H, I).  The workspace (a
    uint8 device tensor) is allocated here when not given."""
    import torch
    n_rows, x_stride = _rows(x, "x")
    H = x.shape[-1]
    if w_gate.dim() != 2 or w_up.shape != w_gate.shape or w_gate.shape[1] != H:
        raise ValueError("w_gate and w_up must both be (I, H)")
    I = w_gate.shape[0]
    if tuple(w_down.shape) != (H, I):
        raise ValueError("w_down must be (H, I)")
    if any(w.dtype != x.dtype for w in (w_gate, w_up, w_down)):
        raise ValueError("x and the weights must have one dtype")
    _, wg_stride = _rows(w_gate, "w_gate")
    _, wu_stride = _rows(w_up, "w_up")
    if wg_stride != wu_stride:
        raise ValueError("w_gate and w_up must have one row stride")
    _, wd_stride = _rows(w_down, "w_down")
    if out is None:
        out = torch.empty(x.shape, dtype=x.dtype, device=x.device)
    _, out_stride = _rows(out, "out")
    code = _dtype_code(x)
    if workspace is None:
        workspace = torch.empty(max(16, glu_mlp_workspace_bytes(max(n_rows, 1), max(I, 1), code)),
                                dtype=torch.uint8, device=x.device)
    st = glu_mlp_fwd(x.data_ptr(), x_stride, w_gate.data_ptr(), w_up.data_ptr(), wg_stride, w_down.data_ptr(),
                     wd_stride, out.data_ptr(), out_stride, n_rows, H, I, ACT[act], code, workspace.data_ptr(),
                     workspace.numel(), _stream(stream))
    if st:
        raise GluError(st, "glu_mlp_fwd")
    return out


def add_rmsnorm(x, residual, gamma, eps: float = 1e-5, *, h=None, y=None, rstd=None, stream=None):
    """h = x + residual and y = rmsnorm(h) * gamma over the last dimension, in one
    pass.  ``h`` and ``y`` may be given (h may be x or residual for an in-place
    residual update, y the other one); ``rstd`` may be a float32 tensor of one
    entry per row, or True to allocate it.  Returns (h, y) or (h, y, rstd)."""
    import torch
    n_rows, x_stride = _rows(x, "x")
    _, r_stride = _rows(residual, "residual")
    if residual.shape != x.shape or residual.dtype != x.dtype:
        raise ValueError("residual must match x in shape and dtype")
    H = x.shape[-1]
    if gamma.shape != (H,) or gamma.dtype != x.dtype or not gamma.is_contiguous():
        raise ValueError("gamma must be a contiguous (H,) tensor of x's dtype")
    h = torch.empty_like(x) if h is None else h
    y = torch.empty_like(x) if y is None else y
    for t, n in ((h, "h"), (y, "y")):
        if t.shape != x.shape or t.dtype != x.dtype:
            raise ValueError(f"{n} must match x in shape and dtype")
    _, h_stride = _rows(h, "h")
    _, y_stride = _rows(y, "y")
    want_rstd = rstd is not None and rstd is not False
    if rstd is True:
        rstd = torch.empty(n_rows, dtype=torch.float32, device=x.device)
    if want_rstd and (rstd.dtype != torch.float32 or rstd.numel() != n_rows or not rstd.is_contiguous()):
        raise ValueError("rstd must be a contiguous float32 tensor with one entry per row")
    st = glu_add_rmsnorm_fwd(x.data_ptr(), x_stride, residual.data_ptr(), r_stride, gamma.data_ptr(),
                             h.data_ptr(), h_stride, y.data_ptr(), y_stride,
                             rstd.data_ptr() if want_rstd else None, n_rows, H, float(eps),
                             _dtype_code(x), _stream(stream))
    if st:
        raise GluError(st, "glu_add_rmsnorm_fwd")
    return (h, y, rstd) if want_rstd else (h, y)


def add_rmsnorm_bwd(dy, h, rstd, gamma, *, dh=None, dx=None, dres=None, dgamma=None, stream=None):
    """Gradients of add_rmsnorm: dx (= the residual's gradient) from dy, the
    stored sum h and rstd, plus dh if h also feeds the residual stream.  ``dres``
    may be a tensor receiving a second copy; ``dgamma`` a float32 (H,) tensor
    the row sums are added to, or True for a zeroed one.  Returns dx, or
    (dx, dgamma) when dgamma is requested."""
    import torch
    n_rows, dy_stride = _rows(dy, "dy")
    _, h_stride = _rows(h, "h")
    H = dy.shape[-1]
    if h.shape != dy.shape or h.dtype != dy.dtype:
        raise ValueError("h must match dy")
    if gamma.shape != (H,) or gamma.dtype != dy.dtype or not gamma.is_contiguous():
        raise ValueError("gamma must be a contiguous (H,) tensor of dy's dtype")
    if rstd.dtype != torch.float32 or rstd.numel() != n_rows or not rstd.is_contiguous():
        raise ValueError("rstd must be a contiguous float32 tensor with one entry per row")
    dx = torch.empty_like(dy) if dx is None else dx
    _, dx_stride = _rows(dx, "dx")
    dh_ptr, dh_stride = (None, 0) if dh is None else (dh.data_ptr(), _rows(dh, "dh")[1])
    dr_ptr, dr_stride = (None, 0) if dres is None else (dres.data_ptr(), _rows(dres, "dres")[1])
    want_dg = dgamma is not None and dgamma is not False
    if dgamma is True:
        dgamma = torch.zeros(H, dtype=torch.float32, device=dy.device)
    if want_dg and (dgamma.dtype != torch.float32 or dgamma.shape != (H,) or not dgamma.is_contiguous()):
        raise ValueError("dgamma must be a contiguous float32 (H,) tensor")
    st = glu_add_rmsnorm_bwd(dy.data_ptr(), dy_stride, h.data_ptr(), h_stride, rstd.data_ptr(), gamma.data_ptr(),
                             dh_ptr, dh_stride, dx.data_ptr(), dx_stride, dr_ptr, dr_stride,
                             dgamma.data_ptr() if want_dg else None, n_rows, H, _dtype_code(dy), _stream(stream))
    if st:
        raise GluError(st, "glu_add_rmsnorm_bwd")
    return (dx, dgamma) if want_dg else dx


# ---- host tensors ---------------------------------------------------------------

def _host_rows(t, name):
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if t.dim() == 1:
        return 1, t.shape[0]
    if t.stride(-1) != 1:
        raise ValueError(f"{name}: the last dimension must be contiguous")
    n = 1
    for s_ in t.shape[:-1]:
        n *= s_
    return n, t.stride(-2)


class HostPipeline:
    """Device workspace and the three streams the host-memory entry points
    use.  Allocation is torch's (plumbing); the copies and kernels are the
    library's."""

    def __init__(self, workspace_bytes: int = 256 << 20, device=None):
        import torch
        dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        self.workspace = torch.empty(workspace_bytes, dtype=torch.uint8, device=dev)
        self.copy_in = torch.cuda.Stream(dev)
        self.copy_out = torch.cuda.Stream(dev)

    def args(self, compute=None):
        import torch
        compute = torch.cuda.current_stream() if compute is None else compute
        return (self.workspace.data_ptr(), self.workspace.numel(), self.copy_in.cuda_stream,
                compute.cuda_stream, self.copy_out.cuda_stream)


def fwd_host(pipe: HostPipeline, a, b=None, *, y=None, act="silu", layout="split", compute=None):
    """glu_fwd_host on CPU tensors (page-locked for overlap).  Returns y (a CPU
    tensor); synchronise the compute stream before reading it."""
    import torch
    concat = layout == "concat"
    n_rows, a_stride = _host_rows(a, "a")
    n_cols = a.shape[-1] // 2 if concat else a.shape[-1]
    if y is None:
        shape = (*a.shape[:-1], n_cols)
        y = torch.empty(shape, dtype=a.dtype, pin_memory=a.is_pinned())
    _, y_stride = _host_rows(y, "y")
    b_ptr, b_stride = (None, 0) if concat else (b.data_ptr(), _host_rows(b, "b")[1])
    st = glu_fwd_host(a.data_ptr(), a_stride, b_ptr, b_stride, y.data_ptr(), y_stride, n_rows, n_cols,
                      LAYOUT[layout], ACT[act], _dtype_code(a), *pipe.args(compute))
    if st:
        raise GluError(st, "glu_fwd_host")
    return y


def bwd_host(pipe: HostPipeline, dc, a, b=None, *, da=None, db=None, act="silu", layout="split",
             compute=None):
    """glu_bwd_host on CPU tensors.  SPLIT returns (da, db); CONCAT returns dx."""
    import torch
    concat = layout == "concat"
    n_rows, a_stride = _host_rows(a, "a")
    _, dc_stride = _host_rows(dc, "dc")
    n_cols = dc.shape[-1]
    pin = a.is_pinned()
    if da is None:
        da = torch.empty(a.shape, dtype=a.dtype, pin_memory=pin)
    _, da_stride = _host_rows(da, "da")
    if concat:
        st = glu_bwd_host(dc.data_ptr(), dc_stride, a.data_ptr(), a_stride, None, 0, da.data_ptr(), da_stride,
                          None, 0, n_rows, n_cols, LAYOUT[layout], ACT[act], _dtype_code(a), *pipe.args(compute))
        if st:
            raise GluError(st, "glu_bwd_host")
        return da
    if db is None:
        db = torch.empty(b.shape, dtype=b.dtype, pin_memory=pin)
    _, b_stride = _host_rows(b, "b")
    _, db_stride = _host_rows(db, "db")
    st = glu_bwd_host(dc.data_ptr(), dc_stride, a.data_ptr(), a_stride, b.data_ptr(), b_stride, da.data_ptr(),
                      da_stride, db.data_ptr(), db_stride, n_rows, n_cols, LAYOUT[layout], ACT[act],
                      _dtype_code(a), *pipe.args(compute))
    if st:
        raise GluError(st, "glu_bwd_host")
    return da, db
