"""GPU parity of glu_add_rmsnorm_fwd (fused residual add + RMSNorm) against the
double-precision oracle, element by element on the same seeded inputs.

The bar: the stored sum h is bit-exact (x + residual in fp32 is exact for
16-bit inputs and correctly rounded for f32, so one rounding either way); y
within 1 ulp of the oracle's exact y rounded once for bf16/f16; for f32,
|y - y_exact| <= 1e-6 |y_exact|: the fp32 sum of squares of non-negative terms
carries at most 21 roundings (partial sums of 8 elements, their pairwise sum,
the warp and block reduction), rstd half of that plus 3 more (divide by H,
add eps, square root and reciprocal), y 2 more, in all at most 14.5 * 2^-24 =
8.6e-7 relative; rstd within 1e-6 relative in every dtype.
Shapes cover 16-byte-vector rows (widths that are multiples of 16 bytes) and
element rows (odd widths, misaligned bases), 16 and 64 elements per thread,
one-warp and 1024-thread blocks, in-place updates and padded strides.
"""
import numpy as np
import pytest
import torch

import glu_activation_mlps_gb300 as glu
import glu_synth
from helpers import TORCH, compare, to_bits, to_dev

pytestmark = pytest.mark.gpu

DTYPES = ("bf16", "f16", "f32")


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    glu.build()
    glu.lib()


def inputs(rows, H, dt, seed, res_sigma=4.0):
    rng = np.random.default_rng([seed, rows, H, DTYPES.index(dt)])
    x = glu_synth.normal_bits(rng, (rows, H), 1.0, dt)
    r = glu_synth.normal_bits(rng, (rows, H), res_sigma, dt)
    g = glu_synth.f32_to_bits(rng.standard_normal(H, dtype=np.float32) * np.float32(0.1) + np.float32(1.0), dt)
    return x, r, g


def check(orc, dt, x, r, g, eps, h_gpu, y_gpu, rstd_gpu, what):
    h, y, rstd, ye = orc.add_rmsnorm(dt, x, r, g, eps)
    assert np.array_equal(h_gpu, h), f"{what}: h differs at {np.flatnonzero(h_gpu != h)[:8]}"
    if dt == "f32":
        compare(y_gpu, y, dt, scale=np.abs(ye), what=what + " y")
    else:
        compare(y_gpu, y, dt, what=what + " y")
    if rstd_gpu is not None:
        rel = np.abs(rstd_gpu.astype(np.float64) - rstd) / rstd
        assert rel.max() <= 1e-6, f"{what}: rstd off by {rel.max():.3g} relative"


def run(x, r, g, dt, eps, want_rstd=True):
    xd, rd, gd = to_dev(x, dt), to_dev(r, dt), to_dev(g, dt)
    h, y, *rest = glu.add_rmsnorm(xd, rd, gd, eps, rstd=True if want_rstd else None)
    torch.cuda.synchronize()
    rstd = rest[0].cpu().numpy() if want_rstd else None
    return to_bits(h, dt), to_bits(y, dt), rstd


SHAPES = [(1, 1), (3, 7), (5, 64), (77, 100), (33, 1000), (64, 4096), (9, 5000), (17, 8192), (4, 16384),
          (3, 16385), (2, 32768), (513, 1536)]


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_parity(orc, shape, dt):
    rows, H = shape
    x, r, g = inputs(rows, H, dt, 1)
    h, y, rstd = run(x, r, g, dt, 1e-5)
    info = glu.glu_last_launch()
    E = 4 if dt == "f32" else 2
    assert info["path"] == 4 and info["vec_bytes"] == (16 if (H * E) % 16 == 0 else E)
    vec = (H * E) % 16 == 0
    persistent = vec and H * E >= 16384 and H <= 1024 * (32 // E)
    assert info["unroll"] == ((32 // E) if persistent else (16 if H <= 16384 else 64))
    assert info["threads"] % 32 == 0 and (info["grid"] <= rows if persistent else info["grid"] == rows)
    check(orc, dt, x, r, g, 1e-5, h, y, rstd, f"{dt} {shape}")


@pytest.mark.parametrize("dt", DTYPES)
def test_eps_and_no_rstd(orc, dt):
    x, r, g = inputs(40, 2048, dt, 2)
    for eps in (1e-6, 0.25, 3.0):
        h, y, _ = run(x, r, g, dt, eps, want_rstd=False)
        check(orc, dt, x, r, g, eps, h, y, None, f"{dt} eps={eps}")


@pytest.mark.parametrize("dt", ("bf16", "f16"))
@pytest.mark.parametrize("mode", ["h=x,y=res", "h=res,y=x"])
def test_in_place(orc, dt, mode):
    """The residual stream updated in place (the usual decoder-block use), with
    y over the other input."""
    rows, H = 300, 4096
    x, r, g = inputs(rows, H, dt, 3)
    xd, rd, gd = to_dev(x, dt), to_dev(r, dt), to_dev(g, dt)
    if mode == "h=x,y=res":
        h, y = glu.add_rmsnorm(xd, rd, gd, 1e-5, h=xd, y=rd)
        assert h.data_ptr() == xd.data_ptr() and y.data_ptr() == rd.data_ptr()
    else:
        h, y = glu.add_rmsnorm(xd, rd, gd, 1e-5, h=rd, y=xd)
    torch.cuda.synchronize()
    check(orc, dt, x, r, g, 1e-5, to_bits(h, dt), to_bits(y, dt), None, f"in place {mode}")


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("offset", [0, 1], ids=["aligned", "misaligned"])
def test_strided_rows_and_guard_bands(orc, dt, offset):
    """Every matrix in rows of H + pad elements starting `offset` elements into a
    NaN-filled buffer: values match the oracle and no byte outside h and y moves."""
    rows, H, pad = 50, 1024, 8
    S = H + pad
    x, r, g = inputs(rows, H, dt, 4)
    T = TORCH[dt]

    def place(bits):
        buf = torch.full((rows * S + offset + 8,), float("nan"), dtype=T, device="cuda")
        view = buf[offset:offset + rows * S].view(rows, S)[:, :H]
        view.copy_(to_dev(bits, dt))
        return buf, view

    _, xv = place(x)
    _, rv = place(r)
    hb, hv = place(np.zeros_like(x))
    yb, yv = place(np.zeros_like(x))
    hb.fill_(float("nan"))
    yb.fill_(float("nan"))
    gd = to_dev(g, dt)
    glu.add_rmsnorm(xv, rv, gd, 1e-5, h=hv, y=yv)
    torch.cuda.synchronize()
    assert glu.glu_last_launch()["vec_bytes"] == (16 if offset == 0 else (4 if dt == "f32" else 2))
    check(orc, dt, x, r, g, 1e-5, to_bits(hv, dt), to_bits(yv, dt), None, f"strided {dt}")
    inside = np.zeros(rows * S + offset + 8, dtype=bool)
    for m in range(rows):
        inside[offset + m * S: offset + m * S + H] = True
    nan_bits = to_bits(torch.full((1,), float("nan"), dtype=T), dt)[0]
    for buf in (hb, yb):
        assert np.all(to_bits(buf, dt)[~inside] == nan_bits)


@pytest.mark.parametrize("dt", DTYPES)
def test_degenerate_rows(orc, dt):
    """All-zero rows give h = 0, rstd = 1/sqrt(eps), y = 0; constant rows give
    y = c / sqrt(c^2 + eps) * gamma; f16 sums beyond 65504 store inf in h while
    y stays finite (the sum and its square are fp32)."""
    H = 256
    x = glu_synth.f32_to_bits(np.zeros((3, H), np.float32), dt)
    r = glu_synth.f32_to_bits(np.zeros((3, H), np.float32), dt)
    x[1] = glu_synth.f32_to_bits(np.full(H, 3.0, np.float32), dt)
    big = 40000.0 if dt == "f16" else 1e5
    x[2] = glu_synth.f32_to_bits(np.full(H, big, np.float32), dt)
    r[2] = glu_synth.f32_to_bits(np.full(H, big, np.float32), dt)
    g = glu_synth.f32_to_bits(np.linspace(0.5, 2.0, H, dtype=np.float32), dt)
    h, y, rstd = run(x, r, g, dt, 1e-5)
    check(orc, dt, x, r, g, 1e-5, h, y, rstd, f"degenerate {dt}")
    assert rstd[0] == pytest.approx(1 / np.sqrt(1e-5), rel=1e-6)


def test_decoder_block_workload(orc):
    """The residual add + RMSNorm of one decoder block at 4096 tokens, hidden
    size 4096, bf16: every element against the oracle."""
    d = glu_synth.add_rmsnorm()
    h, y, rstd = run(d["x"], d["res"], d["gamma"], "bf16", d["eps"])
    check(orc, "bf16", d["x"], d["res"], d["gamma"], d["eps"], h, y, rstd, "decoder block")
