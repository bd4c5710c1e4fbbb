"""Shared helpers for the GPU tests: moving bit arrays to and from the device,
and the comparison bar.

The bar (spec tolerance, read as stated in the design notes):
  * bf16 / f16: the GPU result is within 1 ulp of the oracle's exact result
    rounded once to the dtype.  Ulp distance is the difference of the
    sign-magnitude ordered encodings, so subnormals count as ulps and +0 == -0.
  * f32: |gpu - oracle| <= 1e-6 * max(M, 2^-118), with M = |oracle| for y and
    db and M = |dc*b| * (|t1(a)| + |t2(a)|) for da (the magnitudes of the two
    terms of act'(a), which cancel at the derivative's root).  The floor: every
    result is formed from an exponential; once that exponential is an fp32
    subnormal (below 2^-126) it carries an absolute error of a few 2^-149, which
    the factors a, w'(a) (at most 2^8 there) carry into the result.  Results
    below 2^-118 are therefore held to an absolute error of 1e-6 * 2^-118.
  * NaN must meet NaN.
"""
from __future__ import annotations

import numpy as np
import torch

NP_SIGNED = {"f32": np.int32, "f16": np.int16, "bf16": np.int16}
NP_BITS = {"f32": np.uint32, "f16": np.uint16, "bf16": np.uint16}
TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
TORCH_INT = {"f32": torch.int32, "f16": torch.int16, "bf16": torch.int16}
F32_REL = 1e-6
F32_FLOOR = 2.0 ** -118


def to_dev(bits: np.ndarray, dt: str, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(NP_SIGNED[dt]))
    return t.to(device).view(TORCH[dt])


def to_bits(t: torch.Tensor, dt: str) -> np.ndarray:
    return t.contiguous().view(TORCH_INT[dt]).cpu().numpy().view(NP_BITS[dt])


def ordered16(bits: np.ndarray) -> np.ndarray:
    v = bits.astype(np.int32)
    mag = v & 0x7FFF
    return np.where(v & 0x8000, -mag, mag)


def is_nan(bits: np.ndarray, dt: str) -> np.ndarray:
    if dt == "f32":
        return np.isnan(bits.view(np.float32))
    exp = 0x7C00 if dt == "f16" else 0x7F80
    man = 0x03FF if dt == "f16" else 0x007F
    return ((bits & exp) == exp) & ((bits & man) != 0)


def compare(gpu: np.ndarray, ref: np.ndarray, dt: str, scale: np.ndarray | None = None,
            orc=None, what: str = "") -> dict:
    """Check gpu against ref under the bar; return stats, raise on failure."""
    gpu, ref = np.asarray(gpu).ravel(), np.asarray(ref).ravel()
    assert gpu.shape == ref.shape, what
    gn, rn = is_nan(gpu, dt), is_nan(ref, dt)
    bad_nan = gn != rn
    assert not bad_nan.any(), f"{what}: NaN mismatch at {np.flatnonzero(bad_nan)[:8]}"
    ok = ~rn
    g, r = gpu[ok], ref[ok]
    if dt == "f32":
        gv = g.view(np.float32).astype(np.float64)
        rv = r.view(np.float32).astype(np.float64)
        same_inf = np.isinf(gv) & (gv == rv)
        m = np.abs(rv) if scale is None else np.asarray(scale).ravel()[ok]
        err = np.where(same_inf, 0.0, np.abs(gv - rv))
        tol = F32_REL * np.maximum(m, F32_FLOOR)
        worst = np.argmax(err / tol) if err.size else 0
        stats = {"n": int(err.size), "max_err_over_tol": float((err / tol).max()) if err.size else 0.0,
                 "max_plain_rel": float((err / np.maximum(np.abs(rv), 1e-300)).max()) if err.size else 0.0}
        if err.size and err[worst] > tol[worst]:
            idx = np.flatnonzero(err > tol)
            raise AssertionError(f"{what}: {idx.size} f32 elements outside 1e-6*M; worst gpu={gv[worst]!r} "
                                 f"oracle={rv[worst]!r} M={m[worst]!r} at {np.flatnonzero(ok)[worst]}")
        return stats
    d = np.abs(ordered16(g) - ordered16(r))
    stats = {"n": int(d.size), "max_ulp": int(d.max()) if d.size else 0,
             "frac_off_by_1": float((d == 1).mean()) if d.size else 0.0}
    if d.size and d.max() > 1:
        idx = np.flatnonzero(d > 1)
        raise AssertionError(f"{what}: {idx.size} elements more than 1 ulp off; first at "
                             f"{np.flatnonzero(ok)[idx[:5]]}: gpu={g[idx[:5]]} oracle={r[idx[:5]]}")
    return stats
