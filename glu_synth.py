"""Seeded synthetic inputs for the fused gated activation.

Shared by the tests, the benchmark and the oracle checks.  This module only
draws random numbers and stores them in a dtype's bit pattern; it holds none of
the activation's arithmetic.  Arrays are raw bit patterns: ``uint32`` for f32,
``uint16`` for f16 and bf16 (the bf16 pattern is the top half of the f32 one).

Draws use numpy's PCG64 ``default_rng(seed)`` in float32, scaled by sigma, then
stored in the dtype with round-to-nearest-even.  The workloads are the
intermediate sizes the page "Skill: Write a Triton SiLU-Mul (SwiGLU) Kernel"
lists (Inputs the agent should gather first, item 9) at 4096 tokens, and the
hidden-size sweep of "Kernel Profile: SwiGLU (Tier 1 - Element-wise)"
(Benchmarking).
"""
from __future__ import annotations

import numpy as np

BITS_DTYPE = {"f32": np.uint32, "f16": np.uint16, "bf16": np.uint16}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}


def f32_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Store float32 values in ``dtype`` (round to nearest even)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f32":
        return x.view(np.uint32).copy()
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        u = x.view(np.uint32)
        bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
        return ((u + bias) >> np.uint32(16)).astype(np.uint16)
    raise ValueError(dtype)


def normal_bits(rng: np.random.Generator, shape, sigma: float, dtype: str) -> np.ndarray:
    """i.i.d. N(0, sigma^2) samples stored in ``dtype``."""
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if sigma != 1.0:
        x *= np.float32(sigma)
    return f32_to_bits(x, dtype)


# ---------------------------------------------------------------------------
# Named workloads.  Each returns a dict of bit arrays plus its description.
# ---------------------------------------------------------------------------

def fwd_f32_small(seed: int = 0, rows: int = 256, cols: int = 1024):
    """SwiGLU forward, separate a, b of shape (256, 1024) fp32, a, b ~ N(0, 1)."""
    rng = np.random.default_rng(seed)
    a = normal_bits(rng, (rows, cols), 1.0, "f32")
    b = normal_bits(rng, (rows, cols), 1.0, "f32")
    return {"a": a, "b": b, "dtype": "f32", "act": "silu", "layout": "split"}


def fwd_bf16_split(seed: int = 2, rows: int = 4096, cols: int = 11008):
    """SwiGLU forward, separate a, b (4096, 11008) bf16; a ~ N(0, 2^2), b ~ N(0, 1)."""
    rng = np.random.default_rng(seed)
    a = normal_bits(rng, (rows, cols), 2.0, "bf16")
    b = normal_bits(rng, (rows, cols), 1.0, "bf16")
    return {"a": a, "b": b, "dtype": "bf16", "act": "silu", "layout": "split"}


def fwd_bf16_concat(seed: int = 3, rows: int = 4096, cols: int = 18944):
    """SwiGLU forward on x (4096, 2*18944) bf16, x ~ N(0, 1.5^2); a, b are its halves."""
    rng = np.random.default_rng(seed)
    x = normal_bits(rng, (rows, 2 * cols), 1.5, "bf16")
    return {"x": x, "n_cols": cols, "dtype": "bf16", "act": "silu", "layout": "concat"}


OUTLIER_VALUES = np.array([-88.0, -60.0, -20.0, 20.0, 60.0, 88.0], dtype=np.float32)


def bwd_bf16_outliers(seed: int = 4, rows: int = 4096, cols: int = 28672):
    """SwiGLU backward (4096, 28672) bf16.  a ~ N(0, 3^2) with 1% of entries
    replaced by a uniform pick of +-{20, 60, 88}; b, dc ~ N(0, 1)."""
    rng = np.random.default_rng(seed)
    a32 = rng.standard_normal(size=(rows, cols), dtype=np.float32)
    a32 *= np.float32(3.0)
    mask = rng.random(size=(rows, cols), dtype=np.float32) < np.float32(0.01)
    picks = rng.integers(0, OUTLIER_VALUES.size, size=int(mask.sum()))
    a32[mask] = OUTLIER_VALUES[picks]
    a = f32_to_bits(a32, "bf16")
    del a32
    b = normal_bits(rng, (rows, cols), 1.0, "bf16")
    dc = normal_bits(rng, (rows, cols), 1.0, "bf16")
    return {"a": a, "b": b, "dc": dc, "dtype": "bf16", "act": "silu", "layout": "split"}


SWEEP_H = (1024, 2048, 4096, 8192, 16384)
SWEEP_ACTS = ("silu", "gelu_erf", "gelu_tanh", "relu")
SWEEP_DTYPES = ("bf16", "f16", "f32")


def sweep(H: int, dtype: str, rows: int = 4096, seed: int = 5, with_dc: bool = True):
    """Activation sweep case: a, b, dc (4096, H) i.i.d. N(0, 1) in ``dtype``.
    The seed is derived from (5, H, dtype) so every case is reproducible alone."""
    rng = np.random.default_rng([seed, H, SWEEP_DTYPES.index(dtype)])
    a = normal_bits(rng, (rows, H), 1.0, dtype)
    b = normal_bits(rng, (rows, H), 1.0, dtype)
    out = {"a": a, "b": b, "dtype": dtype, "layout": "split"}
    if with_dc:
        out["dc"] = normal_bits(rng, (rows, H), 1.0, dtype)
    return out


def metric_bf16(seed: int = 6, rows: int = 4096, cols: int = 14336):
    """SwiGLU forward + backward, separate a, b, dc (4096, 14336) bf16, all N(0, 1)."""
    rng = np.random.default_rng(seed)
    a = normal_bits(rng, (rows, cols), 1.0, "bf16")
    b = normal_bits(rng, (rows, cols), 1.0, "bf16")
    dc = normal_bits(rng, (rows, cols), 1.0, "bf16")
    return {"a": a, "b": b, "dc": dc, "dtype": "bf16", "act": "silu", "layout": "split"}


def all_finite_16bit(dtype: str) -> np.ndarray:
    """Every finite bit pattern of a 16-bit dtype (both zeros included)."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    exp_all_ones = (0x7C00 if dtype == "f16" else 0x7F80)
    return bits[(bits & exp_all_ones) != exp_all_ones]


# ---------------------------------------------------------------------------
# Gate/up projections with the activation in the epilogue.
# ---------------------------------------------------------------------------

GRID_EIGHTHS = np.array([-2.0, -1.0, 0.0, 1.0, 2.0], dtype=np.float32) / np.float32(8.0)


def grid_bits(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    """Entries drawn uniformly from {-1/4, -1/8, 0, 1/8, 1/4}: every product is
    a multiple of 2^-6 and every partial sum of up to 2^20 of them is exact in
    fp32, whatever the order of the additions."""
    idx = rng.integers(0, GRID_EIGHTHS.size, size=shape, dtype=np.int8)
    return f32_to_bits(GRID_EIGHTHS[idx], dtype)


def gemm_llama(seed: int = 7, M: int = 4096, K: int = 4096, I: int = 14336, dtype: str = "bf16",
               exact: bool = False):
    """Gate/up projections of one MLP: x (M, K) ~ N(0, 1), w_gate and w_up (I, K)
    ~ N(0, 1/K) (the usual fan-in scale), in ``dtype``.  With ``exact`` every
    operand is drawn from the grid of ``grid_bits`` instead."""
    rng = np.random.default_rng([seed, M, K, I])
    if exact:
        return {"x": grid_bits(rng, (M, K), dtype), "w_gate": grid_bits(rng, (I, K), dtype),
                "w_up": grid_bits(rng, (I, K), dtype), "dtype": dtype}
    s = float(1.0 / np.sqrt(K))
    return {"x": normal_bits(rng, (M, K), 1.0, dtype), "w_gate": normal_bits(rng, (I, K), s, dtype),
            "w_up": normal_bits(rng, (I, K), s, dtype), "dtype": dtype}


# ---------------------------------------------------------------------------
# Residual add + RMSNorm.
# ---------------------------------------------------------------------------

def add_rmsnorm(seed: int = 8, rows: int = 4096, H: int = 4096, dtype: str = "bf16"):
    """One decoder block's residual add + RMSNorm: x (the sub-block's output) ~
    N(0, 1), the residual stream ~ N(0, 4^2) (it grows over the layers),
    gamma ~ 1 + N(0, 0.1^2), eps = 1e-5."""
    rng = np.random.default_rng([seed, rows, H, SWEEP_DTYPES.index(dtype)])
    x = normal_bits(rng, (rows, H), 1.0, dtype)
    res = normal_bits(rng, (rows, H), 4.0, dtype)
    g = rng.standard_normal(size=H, dtype=np.float32) * np.float32(0.1) + np.float32(1.0)
    return {"x": x, "res": res, "gamma": f32_to_bits(g, dtype), "eps": 1e-5, "dtype": dtype}
