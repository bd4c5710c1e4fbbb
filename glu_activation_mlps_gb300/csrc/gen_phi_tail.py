"""Generates the lower-tail normal-CDF approximations used by the GeGLU-erf
kernels (the coefficient tables of `phi_tail` in glu_math.cuh): degree 4 with
C = 0.4 for the forward on bf16 / f16 storage, degree 7 with C = 0.3 for the
backward on bf16 / f16 storage (whose act' amplifies the error of Phi near its
root), degree 10 with C = 0.3 for f32 storage.

For x >= 0 the lower tail of the standard normal distribution is written as

    Phi(-x) = 0.5 * erfc(x / sqrt 2) = exp(-x^2 / 2) * t * P(t),   t = 1 / (1 + C x),

with P a polynomial of degree DEG on t in (0, 1].  P is smooth there: at t = 1
(x = 0) it is 1/2, and as t -> 0 (x -> infinity) it tends to C / sqrt(2 pi),
because Phi(-x) ~ exp(-x^2/2) / (x sqrt(2 pi)) (Mills' ratio).  The exact P is
evaluated with mpmath; the coefficients minimise the maximum relative error
of P by Lawson's iteratively re-weighted least squares on Chebyshev nodes in t,
then are rounded to float32, and the achieved error is re-measured on a dense
grid with the rounded coefficients.

Run:  python glu_activation_mlps_gb300/csrc/gen_phi_tail.py
"""
import mpmath as mp
import numpy as np

C = 0.3
DEG = 7
NODES = 1200
ITERS = 60

mp.mp.dps = 40


def p_exact(t: float) -> float:
    if t == 0.0:
        return float(mp.mpf(C) / mp.sqrt(2 * mp.pi))
    x = (1 / mp.mpf(t) - 1) / mp.mpf(C)
    return float(mp.ncdf(-x) / (mp.e ** (-x * x / 2) * t))


def fit():
    k = np.arange(NODES)
    t = 0.5 - 0.5 * np.cos(np.pi * (k + 0.5) / NODES)
    y = np.array([p_exact(v) for v in t])
    V = np.vander(t, DEG + 1, increasing=True) / y[:, None]     # relative-error rows
    w = np.full(NODES, 1.0 / NODES)
    for _ in range(ITERS):                                      # Lawson: w_i <- w_i |r_i|
        sw = np.sqrt(w)
        coef = np.linalg.lstsq(V * sw[:, None], sw, rcond=None)[0]
        r = np.abs(V @ coef - 1.0)
        w = w * r
        w /= w.sum()
    return coef.astype(np.float32)


def check(coef32):
    t = np.linspace(0.0, 1.0, 40001)
    y = np.array([p_exact(v) for v in t[::4]])
    c64 = coef32.astype(np.float64)
    p64 = np.polynomial.polynomial.polyval(t[::4], c64)
    # float32 Horner with fused multiply-add emulated in float64 then rounded
    p32 = np.full_like(t[::4], np.float32(coef32[-1]), dtype=np.float32)
    for cc in coef32[-2::-1]:
        p32 = (p32.astype(np.float64) * t[::4].astype(np.float32) + np.float64(cc)).astype(np.float32)
    return np.max(np.abs(p64 / y - 1)), np.max(np.abs(p32 / y - 1))


if __name__ == "__main__":
    for c, deg, use in ((0.4, 4, "bf16 / f16 forward"), (0.3, 7, "bf16 / f16 backward"), (0.3, 10, "f32 storage")):
        C, DEG = c, deg
        print(f"// Phi(-x) = exp(-x^2/2) * t * P(t), t = 1/(1 + {C} x)")
        coef = fit()
        e64, e32 = check(coef)
        print(f"// degree {DEG} ({use}): max relative error of P {e64:.2e} with float32 "
              f"coefficients, {e32:.2e} with float32 Horner")
        print("{" + ", ".join(f"{float(v):.9e}f" for v in coef) + "}")
