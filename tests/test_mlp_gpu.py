"""GPU parity of the MLP's second product and of the whole gated MLP.

glu_gemm_nt (d = a b^T, the down projection): on operands from the grid of
glu_synth.grid_bits every partial sum is exact in fp32 whatever the order of
the additions, so every output must be within 1 ulp of the oracle (its one
rounding); on normal inputs the fp32 sums may differ from the exact ones by at
most K 2^-23 sum|products|.

glu_mlp_fwd (out = (act(x wg^T) * (x wu^T)) wd^T, the intermediate y stored
in the dtype): y is held to the 1-ulp bar of glu_gemm_fwd, so out is held to
the propagated bound sum_i ulp(y_i) |wd[h, i]| + I 2^-23 sum_i |y_i wd[h, i]|
plus one output ulp, against the oracle's out of the oracle's y.  Its output
must also equal, bit for bit, glu_gemm_fwd followed by glu_gemm_nt on the same
rows (the same kernels)."""
import numpy as np
import pytest
import torch

import glu_activation_mlps_gb300 as glu
import glu_synth
from helpers import compare, to_bits, to_dev

pytestmark = pytest.mark.gpu

DTYPES = ("bf16", "f16")


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    glu.build()
    glu.lib()


def ulp16(dt, v):
    """The spacing of the dtype's values at |v| (subnormal spacing below the normals)."""
    p, emin = (8, -126) if dt == "bf16" else (11, -14)
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** emin)))
    return 2.0 ** (np.maximum(e, emin) - (p - 1))


def run_nt(a, b, dt, d_stride=None):
    M, K = a.shape
    N = b.shape[0]
    A, B = to_dev(a, dt), to_dev(b, dt)
    ds = d_stride or N
    D = torch.full((M, ds), 7.0, dtype=A.dtype, device="cuda")
    st = glu.glu_gemm_nt(A.data_ptr(), K, B.data_ptr(), K, D.data_ptr(), ds, M, K, N, glu.DTYPE[dt],
                         torch.cuda.current_stream().cuda_stream)
    assert st == 0, glu.glu_status_string(st)
    torch.cuda.synchronize()
    info = glu.glu_last_launch()
    assert info["path"] == 5
    if ds > N:
        assert torch.all(D[:, N:] == 7.0), "padding written"
    return to_bits(D[:, :N], dt)


# (M, K, N): one block (M <= 128), pairs, ragged rows / columns / K steps, each tile width
NT_SHAPES = [(1, 8, 1), (7, 64, 130), (100, 72, 300), (128, 200, 2048), (300, 136, 520), (513, 64, 4096),
             (1024, 16, 8192), (2047, 128, 1000)]


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("shape", NT_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_gemm_nt_grid_inputs_every_output(orc, shape, dt):
    M, K, N = shape
    rng = np.random.default_rng([51, M, K, N, DTYPES.index(dt)])
    a = glu_synth.grid_bits(rng, (M, K), dt)
    b = glu_synth.grid_bits(rng, (N, K), dt)
    d = run_nt(a, b, dt, d_stride=N + (8 if N % 2 else 0))
    mm, nn = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    want, _, _ = orc.matmul_nt_at(dt, a, b, mm.ravel(), nn.ravel())
    compare(d, want.reshape(M, N), dt, what=f"gemm_nt {shape} {dt}")
    assert glu.glu_wait_timeouts() == 0


@pytest.mark.parametrize("dt", DTYPES)
def test_gemm_nt_normal_inputs_accumulation_bound(orc, dt):
    M, K, N = 384, 4096, 1024
    rng = np.random.default_rng(52)
    a = glu_synth.normal_bits(rng, (M, K), 1.0, dt)
    b = glu_synth.normal_bits(rng, (N, K), K ** -0.5, dt)
    d = run_nt(a, b, dt)
    ms, ns = rng.integers(0, M, 3000), rng.integers(0, N, 3000)
    _, ex, sa = orc.matmul_nt_at(dt, a, b, ms, ns)
    got = orc.decode(dt, d[ms, ns])
    allow = K * 2.0 ** -23 * sa + ulp16(dt, np.abs(ex) + K * 2.0 ** -23 * sa)
    assert np.all(np.abs(got - ex) <= allow)


def mlp_inputs(M, H, I, dt, seed, grid=False):
    rng = np.random.default_rng([seed, M, H, I])
    if grid:
        draw = lambda shape: glu_synth.grid_bits(rng, shape, dt)
        return draw((M, H)), draw((I, H)), draw((I, H)), draw((H, I))
    return (glu_synth.normal_bits(rng, (M, H), 1.0, dt), glu_synth.normal_bits(rng, (I, H), H ** -0.5, dt),
            glu_synth.normal_bits(rng, (I, H), H ** -0.5, dt), glu_synth.normal_bits(rng, (H, I), I ** -0.5, dt))


def check_mlp(orc, act, dt, x, wg, wu, wd, out_bits, rows=None, what=""):
    """out against the oracle under the propagated bound; rows: the rows to check (all by default)."""
    if rows is not None:
        x = x[rows]
        out_bits = out_bits[rows]
    want, y, ex, sa = orc.mlp(act, dt, x, wg, wu, wd)
    yv = np.abs(orc.decode(dt, y))
    wdv = np.abs(orc.decode(dt, wd))
    I = wd.shape[1]
    prop = ulp16(dt, yv) @ wdv.T                      # every y_i one ulp off, in the worst direction
    slack = prop + I * 2.0 ** -23 * sa
    allow = slack + ulp16(dt, np.abs(ex) + slack)
    got = orc.decode(dt, out_bits)
    bad = np.flatnonzero(~(np.abs(got - ex) <= allow))
    assert bad.size == 0, (f"{what}: {bad.size} outputs outside the bound; first gpu={got.ravel()[bad[0]]!r} "
                           f"exact={ex.ravel()[bad[0]]!r} allow={allow.ravel()[bad[0]]!r}")
    return float((np.abs(got - ex) / np.maximum(allow, 1e-300)).max())


def run_mlp(x, wg, wu, wd, dt, act, ws_bytes=None):
    X, WG, WU, WD = (to_dev(t, dt) for t in (x, wg, wu, wd))
    M, H = x.shape
    I = wg.shape[0]
    code = glu.DTYPE[dt]
    need = glu.glu_mlp_workspace_bytes(M, I, code)
    ws = torch.empty(ws_bytes or need, dtype=torch.uint8, device="cuda")
    out = torch.empty(M, H, dtype=X.dtype, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = glu.glu_mlp_fwd(X.data_ptr(), H, WG.data_ptr(), WU.data_ptr(), H, WD.data_ptr(), I, out.data_ptr(), H,
                         M, H, I, glu.ACT[act], code, ws.data_ptr(), ws.numel(), s)
    assert st == 0, glu.glu_status_string(st)
    torch.cuda.synchronize()
    return to_bits(out, dt), (X, WG, WU, WD)


MLP_SHAPES = [(1, 64, 72), (77, 128, 304), (300, 256, 1000), (1030, 64, 520)]


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("act", ("silu", "gelu_erf", "gelu_tanh", "relu"))
@pytest.mark.parametrize("shape", MLP_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_mlp_against_oracle_and_composition(orc, shape, act, dt):
    M, H, I = shape
    x, wg, wu, wd = mlp_inputs(M, H, I, dt, 53, grid=(act == "relu"))
    out, (X, WG, WU, WD) = run_mlp(x, wg, wu, wd, dt, act)
    check_mlp(orc, act, dt, x, wg, wu, wd, out, what=f"mlp {shape} {act} {dt}")
    # the same two products called one after the other give the same bits
    y = glu.gemm_fwd(X, WG, WU, act=act)
    d = glu.gemm_nt(y, WD)
    torch.cuda.synchronize()
    assert np.array_equal(to_bits(d, dt), out)
    assert glu.glu_wait_timeouts() == 0


def test_mlp_small_workspace_chunks(orc):
    """A workspace of 3 rows runs 1030 rows in 344 chunks; the result stays
    within the bound (the chunks' tile shapes differ from one call's)."""
    M, H, I = 1030, 64, 104
    x, wg, wu, wd = mlp_inputs(M, H, I, "bf16", 54)
    out, _ = run_mlp(x, wg, wu, wd, "bf16", "silu", ws_bytes=3 * I * 2 + 10)
    check_mlp(orc, "silu", "bf16", x, wg, wu, wd, out, what="mlp chunks of 3 rows")
    out1, _ = run_mlp(x, wg, wu, wd, "bf16", "silu")
    check_mlp(orc, "silu", "bf16", x, wg, wu, wd, out1, what="mlp one chunk")


def test_mlp_full_layer_sampled(orc):
    """One decoder layer's MLP: 4096 tokens, hidden 4096, intermediate 14336,
    bf16, SwiGLU, in one chunk (the default workspace) and in chunks of 1536
    rows; sampled rows (chunk edges among them) against the oracle."""
    M, H, I = 4096, 4096, 14336
    x, wg, wu, wd = mlp_inputs(M, H, I, "bf16", 55)
    out, _ = run_mlp(x, wg, wu, wd, "bf16", "silu")
    rows = np.array([0, 1535, 1536, 2047, 3071, 3072, 4095])
    check_mlp(orc, "silu", "bf16", x, wg, wu, wd, out, rows=rows, what="full layer")
    out2, _ = run_mlp(x, wg, wu, wd, "bf16", "silu", ws_bytes=1536 * I * 2)
    check_mlp(orc, "silu", "bf16", x, wg, wu, wd, out2, rows=rows, what="full layer, 1536-row chunks")
    assert glu.glu_wait_timeouts() == 0
