"""Double-precision CPU oracle for the fused gated activation (test infrastructure).

This package exists to check the CUDA library; it is NOT part of the product
path.  Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it.  It shares no code with the CUDA library and never
imports it.

The arithmetic lives in ``glu_oracle.c`` (plain C, double precision, one RNE
rounding into the storage dtype).  This module compiles it with gcc, loads it
with ctypes, and restates the two operand layouts of the page
"Skill: Write a Triton SiLU-Mul (SwiGLU) Kernel" (Inputs the agent should
gather first, item 4): separate ``a``/``b`` tensors, or one tensor ``x`` whose
row holds ``[gate | up]`` with ``a = x[:, :I]`` and ``b = x[:, I:2I]``.

Arrays are numpy arrays of raw bit patterns: ``uint32`` for f32, ``uint16`` for
f16 and bf16.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "glu_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_glu.so")

ACTS = {"silu": 0, "gelu_erf": 1, "gelu_tanh": 2, "relu": 3}
DTYPES = {"f32": 0, "f16": 1, "bf16": 2}
BITS_DTYPE = {"f32": np.uint32, "f16": np.uint16, "bf16": np.uint16}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, IEEE semantics: no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            i64, vp, dp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
            ci = ctypes.c_int
            L.oracle_fwd.argtypes = [ci, ci, vp, vp, vp, i64]
            L.oracle_bwd.argtypes = [ci, ci, vp, vp, vp, vp, vp, i64]
            L.oracle_bwd_da_scale.argtypes = [ci, ci, vp, vp, vp, dp, i64]
            L.oracle_act_vec.argtypes = [ci, dp, dp, i64]
            L.oracle_act_grad_terms_vec.argtypes = [ci, dp, dp, dp, i64]
            L.oracle_round_vec.argtypes = [ci, dp, dp, i64]
            L.oracle_encode_vec.argtypes = [ci, dp, vp, i64]
            L.oracle_decode_vec.argtypes = [ci, vp, dp, i64]
            L.oracle_gemm_glu_at.argtypes = [ci, ci, vp, i64, vp, vp, i64, i64, vp, vp, i64, vp, dp, dp, dp, dp]
            L.oracle_gemm_glu_at.restype = None
            L.oracle_matmul_nt_at.argtypes = [ci, vp, i64, vp, i64, i64, vp, vp, i64, vp, dp, dp]
            L.oracle_matmul_nt_at.restype = None
            L.oracle_add_rmsnorm.argtypes = [ci, vp, vp, vp, vp, vp, dp, dp, i64, i64, ctypes.c_double]
            L.oracle_add_rmsnorm.restype = None
            L.oracle_add_rmsnorm_bwd.argtypes = [ci, vp, vp, vp, vp, vp, vp, dp, dp, i64, i64]
            L.oracle_add_rmsnorm_bwd.restype = None
            L.oracle_sigmoid.argtypes = [ctypes.c_double]
            L.oracle_sigmoid.restype = ctypes.c_double
            for f in (L.oracle_fwd, L.oracle_bwd, L.oracle_bwd_da_scale, L.oracle_act_vec,
                      L.oracle_act_grad_terms_vec, L.oracle_round_vec, L.oracle_encode_vec,
                      L.oracle_decode_vec):
                f.restype = None
            _lib = L
    return _lib


def _ptr(x: np.ndarray) -> int:
    return x.ctypes.data


def _bits(x, dtype: str) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=BITS_DTYPE[dtype])


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float64)


# ---- scalar maps over doubles -------------------------------------------------

def sigmoid(x: float) -> float:
    return lib().oracle_sigmoid(float(x))


def act(name: str, x) -> np.ndarray:
    """act(x) in double, no rounding."""
    x = _f64(x)
    out = np.empty_like(x)
    lib().oracle_act_vec(ACTS[name], _ptr(x), _ptr(out), x.size)
    return out


def act_grad_terms(name: str, x):
    """The two terms whose sum is act'(x) (see glu_oracle.c)."""
    x = _f64(x)
    t1, t2 = np.empty_like(x), np.empty_like(x)
    lib().oracle_act_grad_terms_vec(ACTS[name], _ptr(x), _ptr(t1), _ptr(t2), x.size)
    return t1, t2


def act_grad(name: str, x) -> np.ndarray:
    t1, t2 = act_grad_terms(name, x)
    return t1 + t2


def round_to(dtype: str, x) -> np.ndarray:
    """Round doubles to the nearest value of ``dtype`` (ties to even)."""
    x = _f64(x)
    out = np.empty_like(x)
    lib().oracle_round_vec(DTYPES[dtype], _ptr(x), _ptr(out), x.size)
    return out


def encode(dtype: str, x) -> np.ndarray:
    x = _f64(x)
    out = np.empty(x.shape, dtype=BITS_DTYPE[dtype])
    lib().oracle_encode_vec(DTYPES[dtype], _ptr(x), _ptr(out), x.size)
    return out


def decode(dtype: str, bits) -> np.ndarray:
    bits = _bits(bits, dtype)
    out = np.empty(bits.shape, dtype=np.float64)
    lib().oracle_decode_vec(DTYPES[dtype], _ptr(bits), _ptr(out), bits.size)
    return out


# ---- element-wise forward / backward over bit arrays --------------------------

def fwd(act_name: str, dtype: str, a, b) -> np.ndarray:
    """y = round(act(a) * b), element by element; a and b have one shape."""
    a, b = _bits(a, dtype), _bits(b, dtype)
    if a.shape != b.shape:
        raise ValueError("a and b must have the same shape")
    y = np.empty_like(a)
    lib().oracle_fwd(ACTS[act_name], DTYPES[dtype], _ptr(a), _ptr(b), _ptr(y), a.size)
    return y


def bwd(act_name: str, dtype: str, dc, a, b):
    """(da, db) = (round(dc * act'(a) * b), round(dc * act(a)))."""
    dc, a, b = _bits(dc, dtype), _bits(a, dtype), _bits(b, dtype)
    if not (a.shape == b.shape == dc.shape):
        raise ValueError("dc, a and b must have the same shape")
    da, db = np.empty_like(a), np.empty_like(a)
    lib().oracle_bwd(ACTS[act_name], DTYPES[dtype], _ptr(dc), _ptr(a), _ptr(b),
                     _ptr(da), _ptr(db), a.size)
    return da, db


def bwd_da_scale(act_name: str, dtype: str, dc, a, b) -> np.ndarray:
    """|dc*b| * (|t1(a)| + |t2(a)|): the magnitude the fp32 da tolerance scales by."""
    dc, a, b = _bits(dc, dtype), _bits(a, dtype), _bits(b, dtype)
    m = np.empty(a.shape, dtype=np.float64)
    lib().oracle_bwd_da_scale(ACTS[act_name], DTYPES[dtype], _ptr(dc), _ptr(a), _ptr(b),
                              _ptr(m), a.size)
    return m


# ---- the concatenated [gate | up] layout --------------------------------------

def split_concat(x, n_cols: int):
    """a = x[:, :I], b = x[:, I:2I] (gate half first)."""
    x = np.asarray(x)
    return x[:, :n_cols], x[:, n_cols:2 * n_cols]


def fwd_concat(act_name: str, dtype: str, x, n_cols: int) -> np.ndarray:
    a, b = split_concat(x, n_cols)
    return fwd(act_name, dtype, a, b)


def bwd_concat(act_name: str, dtype: str, dc, x, n_cols: int) -> np.ndarray:
    """Gradient w.r.t. the concatenated input: dx = [da | db]."""
    a, b = split_concat(x, n_cols)
    da, db = bwd(act_name, dtype, dc, a, b)
    return np.concatenate([da, db], axis=1)


# ---- threaded drivers (the same element-wise calls, split over row blocks) -----

def _row_blocks(n_rows: int, parts: int):
    parts = max(1, min(parts, n_rows))
    step = -(-n_rows // parts)
    return [(r, min(n_rows, r + step)) for r in range(0, n_rows, step)]


def fwd_threaded(act_name: str, dtype: str, a, b, threads: int) -> np.ndarray:
    a, b = _bits(a, dtype), _bits(b, dtype)
    y = np.empty_like(a)
    L, code, dt = lib(), ACTS[act_name], DTYPES[dtype]
    rows = a.reshape(a.shape[0], -1) if a.ndim > 1 else a.reshape(1, -1)
    brow = b.reshape(rows.shape)
    yrow = y.reshape(rows.shape)

    def work(rng):
        r0, r1 = rng
        n = (r1 - r0) * rows.shape[1]
        L.oracle_fwd(code, dt, _ptr(rows[r0:r1]), _ptr(brow[r0:r1]), _ptr(yrow[r0:r1]), n)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(work, _row_blocks(rows.shape[0], threads)))
    return y


def bwd_threaded(act_name: str, dtype: str, dc, a, b, threads: int):
    dc, a, b = _bits(dc, dtype), _bits(a, dtype), _bits(b, dtype)
    da, db = np.empty_like(a), np.empty_like(a)
    L, code, dt = lib(), ACTS[act_name], DTYPES[dtype]
    shp = (a.shape[0], -1) if a.ndim > 1 else (1, -1)
    v = [t.reshape(shp) for t in (dc, a, b, da, db)]

    def work(rng):
        r0, r1 = rng
        n = (r1 - r0) * v[1].shape[1]
        L.oracle_bwd(code, dt, *[_ptr(t[r0:r1]) for t in v], n)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(work, _row_blocks(v[1].shape[0], threads)))
    return da, db


# ---- the gate/up projections with the activation applied ----------------------

def gemm_glu_at(act_name: str, dtype: str, x, w_gate, w_up, ms, is_):
    """y[m, i] = round(act(x[m] . w_gate[i]) * (x[m] . w_up[i])) at the listed
    (m, i) pairs, with the exact (double) g and u and the sums of |products|.
    x is M x K, the weights I x K (bit arrays, row-major, contiguous)."""
    x, wg, wu = _bits(x, dtype), _bits(w_gate, dtype), _bits(w_up, dtype)
    if wg.shape != wu.shape or x.shape[1] != wg.shape[1]:
        raise ValueError("x is M x K and the weights I x K")
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    is_ = np.ascontiguousarray(is_, dtype=np.int64)
    n = ms.size
    y = np.empty(n, dtype=BITS_DTYPE[dtype])
    g, u, sg, su = (np.empty(n) for _ in range(4))
    lib().oracle_gemm_glu_at(ACTS[act_name], DTYPES[dtype], _ptr(x), x.shape[1], _ptr(wg), _ptr(wu),
                             wg.shape[1], x.shape[1], _ptr(ms), _ptr(is_), n, _ptr(y), _ptr(g), _ptr(u),
                             _ptr(sg), _ptr(su))
    return y, g, u, sg, su


def gemm_glu(act_name: str, dtype: str, x, w_gate, w_up):
    """Every output: an M x I bit array (small problems only)."""
    M, I = np.asarray(x).shape[0], np.asarray(w_gate).shape[0]
    mm, ii = np.meshgrid(np.arange(M), np.arange(I), indexing="ij")
    y, *_ = gemm_glu_at(act_name, dtype, x, w_gate, w_up, mm.ravel(), ii.ravel())
    return y.reshape(M, I)


def matmul_nt_at(dtype: str, a, b, ms, ns):
    """d[m, n] = round(a[m] . b[n]) at the listed (m, n) pairs, with the exact
    (double) sums and the sums of |products|.  a is M x K, b is N x K (bit
    arrays, row-major, contiguous)."""
    a, b = _bits(a, dtype), _bits(b, dtype)
    if a.shape[1] != b.shape[1]:
        raise ValueError("a is M x K and b is N x K")
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    n = ms.size
    d = np.empty(n, dtype=BITS_DTYPE[dtype])
    ex, sa = np.empty(n), np.empty(n)
    lib().oracle_matmul_nt_at(DTYPES[dtype], _ptr(a), a.shape[1], _ptr(b), b.shape[1], a.shape[1],
                              _ptr(ms), _ptr(ns), n, _ptr(d), _ptr(ex), _ptr(sa))
    return d, ex, sa


def mlp(act_name: str, dtype: str, x, w_gate, w_up, w_down):
    """The gated MLP, every output: y = round(act(x w_gate^T) * (x w_up^T)),
    the intermediate stored in the dtype, then out = round(y w_down^T), with
    the exact (double) down sums and their sums of |products| (small problems
    only).  w_down is H x I (row h holds output feature h)."""
    y = gemm_glu(act_name, dtype, x, w_gate, w_up)
    M, H = y.shape[0], np.asarray(w_down).shape[0]
    mm, hh = np.meshgrid(np.arange(M), np.arange(H), indexing="ij")
    d, ex, sa = matmul_nt_at(dtype, y, w_down, mm.ravel(), hh.ravel())
    return d.reshape(M, H), y, ex.reshape(M, H), sa.reshape(M, H)


# ---- fused residual add + RMSNorm --------------------------------------------

def add_rmsnorm(dtype: str, x, res, gamma, eps: float):
    """h = x + res (exact, stored rounded), y = round(h * rstd * gamma) with
    rstd = 1 / sqrt(mean(h^2) + eps) over each row of the exact h.  x and res
    are (rows, H) bit arrays, gamma (H,).  Returns (h, y, rstd, y_exact)."""
    x, res = _bits(x, dtype), _bits(res, dtype)
    gamma = _bits(gamma, dtype)
    if x.ndim != 2 or res.shape != x.shape or gamma.shape != (x.shape[1],):
        raise ValueError("x and res are (rows, H), gamma is (H,)")
    rows, H = x.shape
    h, y = np.empty_like(x), np.empty_like(x)
    rstd = np.empty(rows)
    y_exact = np.empty((rows, H))
    lib().oracle_add_rmsnorm(DTYPES[dtype], _ptr(x), _ptr(res), _ptr(gamma), _ptr(h), _ptr(y), _ptr(rstd),
                             _ptr(y_exact), rows, H, float(eps))
    return h, y, rstd, y_exact


def add_rmsnorm_bwd(dtype: str, dy, h, rstd, gamma, dh=None):
    """ds = rstd*gamma*dy - (rstd^3/H) * h * sum(gamma*dy*h) (+ dh), rounded once,
    and dgamma = sum over rows of dy*h*rstd.  dy, h (and dh) are (rows, H) bit
    arrays, rstd a float32 array of one value per row, gamma (H,) bits.
    Returns (ds bits, ds exact, dgamma)."""
    dy, h, gamma = _bits(dy, dtype), _bits(h, dtype), _bits(gamma, dtype)
    rstd = np.ascontiguousarray(rstd, dtype=np.float32)
    if dy.ndim != 2 or h.shape != dy.shape or rstd.shape != (dy.shape[0],) or gamma.shape != (dy.shape[1],):
        raise ValueError("dy, h are (rows, H), rstd (rows,), gamma (H,)")
    rows, H = dy.shape
    if dh is not None:
        dh = _bits(dh, dtype)
        if dh.shape != dy.shape:
            raise ValueError("dh must match dy")
    ds = np.empty_like(dy)
    ds_exact = np.empty((rows, H))
    dgamma = np.empty(H)
    lib().oracle_add_rmsnorm_bwd(DTYPES[dtype], _ptr(dy), _ptr(h), _ptr(rstd), _ptr(gamma),
                                 _ptr(dh) if dh is not None else None, _ptr(ds), _ptr(ds_exact), _ptr(dgamma),
                                 rows, H)
    return ds, ds_exact, dgamma
