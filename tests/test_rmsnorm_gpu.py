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

The backward (glu_add_rmsnorm_bwd) is held to a bound derived from its fp32
arithmetic (check_bwd) on the same kinds of rows: the staged kernel with a
producer warp (up to 1024 16-byte vectors a row) and without one (wider
rows), the element kernel, ragged stages, in place, a second output, and
pinned host inputs.
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


# ---------------------------------------------------------------- backward
# ds (dx, dres) against the oracle's exact value: the fp32 path may differ by
# E = 32 * 2^-24 * (|rstd gamma dy| + rstd^3 / H * sum_k |gamma dy s| * |s| + |dh|)
# (the row sum carries at most 21 roundings of its terms' magnitudes, rstd^3/H a
# few more, each product and sum one), then one rounding into the dtype.
# dgamma: one fused multiply-add per row per block and one atomic addition per
# block, at most (rows + blocks) roundings of sum_r |dy s rstd|.

U = 2.0 ** -24


def ulp(dt, v):
    v = np.abs(np.asarray(v, dtype=np.float64))
    lo, p = {"bf16": (-126, 7), "f16": (-14, 10), "f32": (-126, 23)}[dt]
    e = np.floor(np.log2(np.maximum(v, 2.0 ** lo)))
    return 2.0 ** (np.maximum(e, lo) - p)


def bwd_inputs(rows, H, dt, seed, with_dh):
    rng = np.random.default_rng([seed, rows, H, DTYPES.index(dt), int(with_dh)])
    h = glu_synth.normal_bits(rng, (rows, H), 3.0, dt)
    dy = glu_synth.normal_bits(rng, (rows, H), 1.0, dt)
    g = glu_synth.f32_to_bits(rng.standard_normal(H, dtype=np.float32) * np.float32(0.2) + np.float32(1.0), dt)
    rstd = (rng.random(rows, dtype=np.float32) * np.float32(0.5) + np.float32(0.2)).astype(np.float32)
    dh = glu_synth.normal_bits(rng, (rows, H), 0.5, dt) if with_dh else None
    return dy, h, rstd, g, dh


def check_bwd(orc, dt, dy, h, rstd, g, dh, dx_gpu, dg_gpu, what, n_blocks=5000):
    _, ds, dgamma = orc.add_rmsnorm_bwd(dt, dy, h, rstd, g, dh)
    d, s, gv = orc.decode(dt, dy), orc.decode(dt, h), orc.decode(dt, g)
    rs = rstd.astype(np.float64)[:, None]
    H = d.shape[1]
    big = np.sum(np.abs(gv[None, :] * d * s), axis=1, keepdims=True)
    E = 32 * U * (np.abs(rs * gv[None, :] * d) + rs ** 3 / H * big * np.abs(s) +
                  (np.abs(orc.decode(dt, dh)) if dh is not None else 0.0))
    got = orc.decode(dt, dx_gpu)
    allow = E + ulp(dt, np.abs(ds) + E)
    bad = np.flatnonzero(~(np.abs(got - ds) <= allow))
    assert bad.size == 0, (f"{what}: {bad.size} ds outside the bound; first {bad[0]}: gpu {got.ravel()[bad[0]]!r} "
                           f"exact {ds.ravel()[bad[0]]!r} allow {allow.ravel()[bad[0]]!r}")
    if dg_gpu is not None:
        rows = d.shape[0]
        scale = np.sum(np.abs(d * s * rs), axis=0)
        err = np.abs(dg_gpu.astype(np.float64) - dgamma)
        assert np.all(err <= (rows + n_blocks) * U * scale + 1e-30), f"{what}: dgamma off by {err.max():.3g}"


def run_bwd(dy, h, rstd, g, dh, dt, dres=False, dgamma=True):
    dyd, hd, gd = to_dev(dy, dt), to_dev(h, dt), to_dev(g, dt)
    rd = torch.from_numpy(rstd).cuda()
    dhd = to_dev(dh, dt) if dh is not None else None
    dr = torch.empty_like(dyd) if dres else None
    out = glu.add_rmsnorm_bwd(dyd, hd, rd, gd, dh=dhd, dres=dr, dgamma=True if dgamma else None)
    torch.cuda.synchronize()
    dx, dg = out if dgamma else (out, None)
    if dres:
        assert torch.equal(dr.view(TORCH_INT_OF[dt]), dx.view(TORCH_INT_OF[dt]))
    return to_bits(dx, dt), (dg.cpu().numpy() if dg is not None else None)


TORCH_INT_OF = {"bf16": torch.int16, "f16": torch.int16, "f32": torch.int32}
# (30011, 64) and (6000, 1024): the persistent team kernel with several rows
# per team; (3001, 6144): stages that go round the shared-memory ring of the
# staged kernel several times, the last one ragged; (9, 5000): a
# 160-thread team beside the producer warp; (33, 8200): just past 1024
# vectors a row (16-bit types), the kernel without a producer warp on a
# 288-thread team; (5000, 1000): the persistent team kernel with the last
# vectors of a row past some threads' reach (125 and 250 vectors a row);
# (64, 4096): 512 vectors, the widest rows of the team kernel for 16-bit
# types and past it for f32
BWD_SHAPES = [(1, 1), (3, 7), (5, 64), (77, 100), (33, 1000), (64, 4096), (9, 5000), (17, 8192), (4, 16384),
              (513, 1536), (30011, 64), (6000, 1024), (33, 8200), (5000, 1000), (3001, 6144)]


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("shape", BWD_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_bwd_parity(orc, shape, dt):
    rows, H = shape
    for with_dh, dres in ((False, False), (True, True)):
        dy, h, rstd, g, dh = bwd_inputs(rows, H, dt, 20, with_dh)
        dx, dg = run_bwd(dy, h, rstd, g, dh, dt, dres=dres)
        info = glu.glu_last_launch()
        E = 4 if dt == "f32" else 2
        V = 16 // E
        vec = (H * E) % 16 == 0 and H <= 2048 * V
        assert info["backward"] == 1 and info["vec_bytes"] == (16 if vec else E) and info["grid"] <= rows
        nvec = H // V
        if not vec:
            assert info["path"] == 4
            nv = 0
        elif info["path"] == 7:
            # the narrow kernel: one 16-byte access per operand per thread and row, rows of up to 128
            assert nvec <= 128 and info["threads"] == 256
            nv = 1
        elif nvec <= (512 if E == 2 else 384):
            # the persistent team kernel: 4 accesses per operand per thread where every lane of a warp
            # has 4 (at most 2 with dh), else 2 or 1; whole teams of whole warps, at most 1024 threads
            assert info["path"] == 8
            nv = 4 if nvec >= 128 else 2 if nvec >= 64 else 1
            nv = min(nv, 2) if with_dh else nv
            tpr = (-(-nvec // nv) + 31) // 32 * 32
            assert info["threads"] % tpr == 0 and info["threads"] <= 1024
        else:
            # the staged kernel: the fewest accesses (2 or 4) that keep a row within 256 consumer
            # threads beside the producer warp; wider rows 4 at 512 threads
            assert info["path"] == 6
            nv = 2 if H <= 512 * V else 4
        assert info["unroll"] == (nv * V if vec else 16)
        assert glu.glu_wait_timeouts() == 0
        check_bwd(orc, dt, dy, h, rstd, g, dh, dx, dg, f"bwd {dt} {shape} dh={with_dh}")


@pytest.mark.parametrize("dt", ("bf16", "f32"))
def test_bwd_in_place_and_accumulation(orc, dt):
    """dx over dy and dres over h; then dx over dh; dgamma adds to what it holds."""
    rows, H = 300, 2048
    dy, h, rstd, g, dh = bwd_inputs(rows, H, dt, 21, True)
    dyd, hd, gd, dhd = to_dev(dy, dt), to_dev(h, dt), to_dev(g, dt), to_dev(dh, dt)
    rd = torch.from_numpy(rstd).cuda()
    dg = torch.zeros(H, dtype=torch.float32, device="cuda")
    glu.add_rmsnorm_bwd(dyd, hd, rd, gd, dh=dhd, dx=dyd, dres=hd, dgamma=dg)
    torch.cuda.synchronize()
    check_bwd(orc, dt, dy, h, rstd, g, dh, to_bits(dyd, dt), dg.cpu().numpy(), "in place over dy")
    assert torch.equal(dyd.view(TORCH_INT_OF[dt]), hd.view(TORCH_INT_OF[dt]))
    # a second call over the untouched originals, dx over dh, adds the same dgamma again
    dyd, hd, dhd = to_dev(dy, dt), to_dev(h, dt), to_dev(dh, dt)
    glu.add_rmsnorm_bwd(dyd, hd, rd, gd, dh=dhd, dx=dhd, dgamma=dg)
    torch.cuda.synchronize()
    check_bwd(orc, dt, dy, h, rstd, g, dh, to_bits(dhd, dt), dg.cpu().numpy() / 2, "in place over dh")


def test_forward_then_backward_decoder_block(orc):
    """The training step's pair on the decoder-block workload: the forward's h
    and rstd feed the backward; every element against the oracle given the same
    h and rstd."""
    d = glu_synth.add_rmsnorm()
    rows, H = d["x"].shape
    xd, rd_, gd = to_dev(d["x"], "bf16"), to_dev(d["res"], "bf16"), to_dev(d["gamma"], "bf16")
    h, y, rstd = glu.add_rmsnorm(xd, rd_, gd, d["eps"], rstd=True)
    rng = np.random.default_rng(22)
    dy = glu_synth.normal_bits(rng, (rows, H), 1.0, "bf16")
    dx, dg = glu.add_rmsnorm_bwd(to_dev(dy, "bf16"), h, rstd, gd, dgamma=True)
    torch.cuda.synchronize()
    check_bwd(orc, "bf16", dy, to_bits(h, "bf16"), rstd.cpu().numpy(), d["gamma"], None, to_bits(dx, "bf16"),
              dg.cpu().numpy(), "decoder block backward")


@pytest.mark.parametrize("dt", ("bf16", "f32"))
def test_pinned_host_memory(orc, dt):
    """Both entry points on pinned host buffers, through the C calls (the
    kernels read and write them in place over the host link): the forward on
    its 16-byte path, the backward on element accesses (its staged kernel takes
    device-memory inputs only).  dgamma must be in device memory: pinned host
    memory there is refused before any launch."""
    rows, H = 300, 1024
    code, T = {"bf16": (2, torch.bfloat16), "f32": (0, torch.float32)}[dt]
    pin = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(
        {"bf16": np.int16, "f32": np.int32}[dt])).view(T).pin_memory()
    s = torch.cuda.current_stream().cuda_stream
    E = 4 if dt == "f32" else 2

    x, r, g = inputs(rows, H, dt, 31)
    X, RES, GAM = pin(x), pin(r), pin(g)
    Hh, Y = (torch.empty(rows, H, dtype=T).pin_memory() for _ in range(2))
    RSTD = torch.empty(rows, dtype=torch.float32).pin_memory()
    assert glu.glu_add_rmsnorm_fwd(X.data_ptr(), H, RES.data_ptr(), H, GAM.data_ptr(), Hh.data_ptr(), H,
                                   Y.data_ptr(), H, RSTD.data_ptr(), rows, H, 1e-5, code, s) == 0
    torch.cuda.synchronize()
    assert glu.glu_last_launch()["vec_bytes"] == 16
    check(orc, dt, x, r, g, 1e-5, to_bits(Hh, dt), to_bits(Y, dt), RSTD.numpy(), "pinned forward")

    dy, h, rstd, g2, dh = bwd_inputs(rows, H, dt, 32, True)
    DY, HH, G2, DH = pin(dy), pin(h), pin(g2), pin(dh)
    RS = torch.from_numpy(rstd).pin_memory()
    DX = torch.empty(rows, H, dtype=T).pin_memory()
    dg = torch.zeros(H, dtype=torch.float32, device="cuda")
    assert glu.glu_add_rmsnorm_bwd(DY.data_ptr(), H, HH.data_ptr(), H, RS.data_ptr(), G2.data_ptr(), DH.data_ptr(),
                                   H, DX.data_ptr(), H, None, 0, dg.data_ptr(), rows, H, code, s) == 0
    torch.cuda.synchronize()
    assert glu.glu_last_launch()["vec_bytes"] == E
    check_bwd(orc, dt, dy, h, rstd, g2, dh, to_bits(DX, dt), dg.cpu().numpy(), "pinned backward")

    DG = torch.zeros(H, dtype=torch.float32).pin_memory()
    assert glu.glu_add_rmsnorm_bwd(DY.data_ptr(), H, HH.data_ptr(), H, RS.data_ptr(), G2.data_ptr(), None, 0,
                                   DX.data_ptr(), H, None, 0, DG.data_ptr(), rows, H, code, s) == -8   # GLU_ERR_VALUE
