"""GPU parity of glu_gemm_fwd (gate/up projections with the activation in the
epilogue, on the tensor cores) against the double-precision oracle.

Two bars:
  * grid inputs (every entry in {-1/4, -1/8, 0, 1/8, 1/4}): g and u are exact in
    fp32 whatever order the tensor cores add in, so y must be within 1 ulp of
    the oracle's y (the same bar as the streaming kernels);
  * normal inputs: the fp32 sums differ from the exact ones by at most
    K * 2^-23 * S (S = the sum of |products|; the bound allows truncating adds),
    and the activation is 1.2-Lipschitz, so y may differ from act(g) * u by that
    propagated error, plus 1e-5 relative for the fp32 activation, plus one ulp of
    the final rounding.
Shapes span several 128 x 128 tiles with ragged M, I and K; padded strides
check that nothing beyond K is read; a misaligned, strided y takes the
element-wise store path.  The full projection of one MLP layer (M = 4096,
K = 4096, I = 14336) is checked on sampled outputs.
"""
import numpy as np
import pytest
import torch

import glu_activation_mlps_gb300 as glu
import glu_synth
from helpers import TORCH, compare, to_bits, to_dev

pytestmark = pytest.mark.gpu

ACTS = ("silu", "gelu_erf", "gelu_tanh", "relu")
DTYPES = ("bf16", "f16")
LIPSCHITZ = 1.2      # |act(s) - act(t)| <= 1.2 |s - t| for all four activations


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    glu.build()
    glu.lib()
    glu.glu_wait_timeouts(reset=True)
    yield
    torch.cuda.synchronize()
    assert glu.glu_wait_timeouts() == 0


def ulp16(dt, v):
    v = np.abs(np.asarray(v, dtype=np.float64))
    lo, p = (-126, 7) if dt == "bf16" else (-14, 10)
    e = np.floor(np.log2(np.maximum(v, 2.0 ** lo)))
    return 2.0 ** (np.maximum(e, lo) - p)


def padded(bits, stride, fill):
    """Copy a (rows, K) bit array into rows of `stride` elements, the pad set to `fill`."""
    rows, K = bits.shape
    out = np.full((rows, stride), fill, dtype=bits.dtype)
    out[:, :K] = bits
    return out


def run_gemm(x, wg, wu, dt, act, K, y_stride=None, y_offset=0):
    """Launch through the C entry point with explicit strides; return y bits (M, I)."""
    M, I = x.shape[0], wg.shape[0]
    xd, gd, ud = to_dev(x, dt), to_dev(wg, dt), to_dev(wu, dt)
    ys = I if y_stride is None else y_stride
    ybuf = torch.full((M * ys + y_offset + 8,), float("nan"), dtype=xd.dtype, device="cuda")
    st = glu.glu_gemm_fwd(xd.data_ptr(), x.shape[1], gd.data_ptr(), ud.data_ptr(), wg.shape[1],
                          ybuf.data_ptr() + 2 * y_offset, ys, M, K, I, glu.ACT[act], glu.DTYPE[dt],
                          torch.cuda.current_stream().cuda_stream)
    assert st == 0, glu.glu_status_string(st)
    torch.cuda.synchronize()
    y = ybuf[y_offset:y_offset + M * ys].view(M, ys)
    return to_bits(y[:, :I], dt), to_bits(ybuf, dt), ys


def check_bound(orc, act, dt, y_bits, g, u, sg, su, K, what):
    ex = orc.act(act, g) * u
    dg = K * 2.0 ** -23 * sg
    du = K * 2.0 ** -23 * su
    slack = LIPSCHITZ * np.abs(u) * dg + np.abs(orc.act(act, g)) * du + LIPSCHITZ * dg * du
    allow = slack + 1e-5 * np.abs(ex) + ulp16(dt, np.abs(ex) + slack)
    yv = orc.decode(dt, y_bits).ravel()
    err = np.abs(yv - ex)
    bad = np.flatnonzero(~(err <= allow))
    assert bad.size == 0, (f"{what}: {bad.size} outputs outside the accumulation bound; first at {bad[0]}: "
                           f"gpu={yv[bad[0]]!r} exact={ex[bad[0]]!r} allow={allow[bad[0]]!r}")
    return float((err / np.maximum(allow, 1e-300)).max())


# ---------------------------------------------------------------- exact grid inputs, every output

# M <= 128 runs one block per tile, larger M pairs of blocks on 256 rows;
# column tiles are 64, 96 or 128 wide (the rule in expected_tiles), and the
# shapes below take each width in both block shapes: one block 96 at
# (5, 520, 14336) and 128 at (100, 64, 38912); pairs 96 at (256, 64, 14336)
# and 128 at (700, 16, 14336) and (1024, 16, 14336); 64 elsewhere.  A ragged
# last row block whose second block reads no row at all (1100, 72, 300), and
# ragged rows and columns (2047, 136, 520).
SHAPES = [(1, 8, 1), (128, 64, 128), (127, 72, 65), (300, 200, 300), (129, 1000, 40), (257, 328, 200),
          (64, 4096, 64), (700, 256, 520), (333, 136, 100), (5, 520, 14336), (256, 64, 14336),
          (100, 64, 38912), (700, 16, 14336), (1024, 16, 14336), (1100, 72, 300), (2047, 136, 520)]


def cluster_size(M, I):
    return 1 if M <= 128 else 2


def expected_tiles(M, I, sms):
    """The library's tile-width rule: the width in {128, 96, 64} whose rounds of
    tiles (ceil(tiles / slots) of them) move the fewest operand rows per K step
    (a tile's rows of x, 256 for a pair or M rounded up to 8 for one block, plus
    2 x width rows of weights), the widest on a tie; 64 when I fits one tile."""
    ctas = cluster_size(M, I)
    m_blocks = -(-M // (128 * ctas))
    slots = sms // ctas
    a_rows = 256 if ctas == 2 else -(-M // 8) * 8
    if I <= 64:
        return m_blocks
    best = None
    for bn in (128, 96, 64):
        tiles = m_blocks * -(-I // bn)
        cost = -(-tiles // slots) * (a_rows + 2 * bn)
        if best is None or cost < best[0]:
            best = (cost, tiles)
    return best[1]


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_grid_inputs_every_output(orc, shape, act, dt):
    M, K, I = shape
    rng = np.random.default_rng([11, M, K, I, ACTS.index(act), DTYPES.index(dt)])
    x = glu_synth.grid_bits(rng, (M, K), dt)
    wg = glu_synth.grid_bits(rng, (I, K), dt)
    wu = glu_synth.grid_bits(rng, (I, K), dt)
    y, _, _ = run_gemm(x, wg, wu, dt, act, K)
    info = glu.glu_last_launch()
    assert info["path"] == 3 and info["unroll"] == cluster_size(M, I) and info["grid"] % info["unroll"] == 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert info["vector_units"] == expected_tiles(M, I, sms)
    ref = orc.gemm_glu(act, dt, x, wg, wu)
    compare(y, ref, dt, what=f"gemm {act} {dt} {shape}")


@pytest.mark.parametrize("dt", DTYPES)
def test_many_tiles_per_block(orc, dt):
    """More tiles than resident blocks: each block (or pair) walks several
    tiles, alternating its two tensor-memory accumulators."""
    M, K, I = 1536, 64, 6144
    rng = np.random.default_rng(17)
    x = glu_synth.grid_bits(rng, (M, K), dt)
    wg = glu_synth.grid_bits(rng, (I, K), dt)
    wu = glu_synth.grid_bits(rng, (I, K), dt)
    y, _, _ = run_gemm(x, wg, wu, dt, "gelu_erf", K)
    compare(y, orc.gemm_glu("gelu_erf", dt, x, wg, wu), dt, what="many tiles")


# ---------------------------------------------------------------- normal inputs, accumulation bound

@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("shape", [(256, 4096, 384), (200, 1000, 130)], ids=lambda s: "x".join(map(str, s)))
def test_normal_inputs_accumulation_bound(orc, shape, act, dt):
    M, K, I = shape
    d = glu_synth.gemm_llama(seed=12, M=M, K=K, I=I, dtype=dt)
    y, _, _ = run_gemm(d["x"], d["w_gate"], d["w_up"], dt, act, K)
    mm, ii = np.meshgrid(np.arange(M), np.arange(I), indexing="ij")
    _, g, u, sg, su = orc.gemm_glu_at(act, dt, d["x"], d["w_gate"], d["w_up"], mm.ravel(), ii.ravel())
    check_bound(orc, act, dt, y, g, u, sg, su, K, f"gemm {act} {dt} {shape}")


# ---------------------------------------------------------------- strides, padding, store paths

@pytest.mark.parametrize("I,y_stride,y_offset,store", [(77, 82, 1, 2), (77, 88, 0, 16), (80, 88, 0, 64)],
                         ids=["misaligned", "aligned-ragged-width", "aligned"])
@pytest.mark.parametrize("dt", DTYPES)
def test_padded_operands_and_strided_output(orc, dt, I, y_stride, y_offset, store):
    """K = 20 is not a multiple of the 64-wide K slice nor of 8: the operands
    live in rows of 24 elements whose pad holds 1e4 (never read: the copy
    engine zero-fills beyond K).  y has I columns in rows of y_stride: one
    element past a 16-byte boundary (element stores), 16-byte aligned with a
    width that is not (16-byte stores from registers), or aligned throughout
    (boxes through the copy engine, clipped at column I and row M).  The words
    around y must stay untouched."""
    M, K, S = 150, 20, 24
    rng = np.random.default_rng(13)
    big = glu_synth.f32_to_bits(np.array([1e4], dtype=np.float32), dt)[0]
    x = glu_synth.grid_bits(rng, (M, K), dt)
    wg = glu_synth.grid_bits(rng, (I, K), dt)
    wu = glu_synth.grid_bits(rng, (I, K), dt)
    y, ybuf, ys = run_gemm(padded(x, S, big), padded(wg, S, big), padded(wu, S, big), dt, "silu", K,
                           y_stride=y_stride, y_offset=y_offset)
    assert glu.glu_last_launch()["vec_bytes"] == store
    compare(y, orc.gemm_glu("silu", dt, x, wg, wu), dt, what="padded")
    # the gaps between y's rows and the words before and after it are still NaN
    inside = np.zeros(ybuf.size, dtype=bool)
    for m in range(M):
        inside[y_offset + m * ys: y_offset + m * ys + I] = True
    nan_bits = to_bits(torch.full((1,), float("nan"), dtype=TORCH[dt]), dt)[0]
    assert np.all(ybuf[~inside] == nan_bits)


@pytest.mark.parametrize("dt", DTYPES)
def test_tensor_helper_matches_entry_point(orc, dt):
    """gemm_fwd on torch tensors (3-D x, weights in the nn.Linear layout)."""
    rng = np.random.default_rng(14)
    B, T, K, I = 2, 70, 136, 190
    x = glu_synth.grid_bits(rng, (B * T, K), dt)
    wg = glu_synth.grid_bits(rng, (I, K), dt)
    wu = glu_synth.grid_bits(rng, (I, K), dt)
    y = glu.gemm_fwd(to_dev(x, dt).view(B, T, K), to_dev(wg, dt), to_dev(wu, dt), act="gelu_tanh")
    assert y.shape == (B, T, I)
    compare(to_bits(y.reshape(B * T, I), dt), orc.gemm_glu("gelu_tanh", dt, x, wg, wu), dt, what="helper")


def test_degenerate_sizes():
    dev = "cuda"
    x = torch.zeros(4, 16, dtype=torch.bfloat16, device=dev)
    w = torch.zeros(8, 16, dtype=torch.bfloat16, device=dev)
    y = torch.full((4, 8), 3.0, dtype=torch.bfloat16, device=dev)
    s = torch.cuda.current_stream().cuda_stream
    # K == 0: empty sums, y = act(0) * 0 = 0 for every activation
    for act in ACTS:
        y.fill_(3.0)
        assert glu.glu_gemm_fwd(x.data_ptr(), 16, w.data_ptr(), w.data_ptr(), 16, y.data_ptr(), 8,
                                4, 0, 8, glu.ACT[act], glu.DTYPE["bf16"], s) == 0
        torch.cuda.synchronize()
        assert torch.all(y == 0)
    # M == 0 or I == 0: nothing is written
    y.fill_(3.0)
    assert glu.glu_gemm_fwd(x.data_ptr(), 16, w.data_ptr(), w.data_ptr(), 16, y.data_ptr(), 8,
                            0, 16, 8, 0, glu.DTYPE["bf16"], s) == 0
    assert glu.glu_gemm_fwd(x.data_ptr(), 16, w.data_ptr(), w.data_ptr(), 16, y.data_ptr(), 8,
                            4, 16, 0, 0, glu.DTYPE["bf16"], s) == 0
    torch.cuda.synchronize()
    assert torch.all(y == 3.0)


def test_against_torch_matmul():
    """A sanity check beside the oracle: torch's fp32 matmul then the same
    formula in fp32 agree with the fused result to bf16 precision."""
    torch.manual_seed(15)
    M, K, I = 512, 1024, 768
    x = torch.randn(M, K, device="cuda").bfloat16()
    wg = (torch.randn(I, K, device="cuda") / K ** 0.5).bfloat16()
    wu = (torch.randn(I, K, device="cuda") / K ** 0.5).bfloat16()
    y = glu.gemm_fwd(x, wg, wu, act="silu").float()
    g, u = x.float() @ wg.float().T, x.float() @ wu.float().T
    ref = torch.nn.functional.silu(g) * u
    assert torch.allclose(y, ref, rtol=2 ** -7, atol=1e-3)


# ---------------------------------------------------------------- one MLP layer at full size, sampled

def sample_positions(M, I, n, seed):
    rng = np.random.default_rng(seed)
    ms = np.concatenate([rng.integers(0, M, n), [0, M - 1, 127, 128, M - 1, 0]])
    is_ = np.concatenate([rng.integers(0, I, n), [0, I - 1, 127, 128, 0, I - 1]])
    return ms, is_


@pytest.mark.parametrize("exact", [True, False], ids=["grid", "normal"])
def test_full_layer_sampled(orc, exact):
    M, K, I = 4096, 4096, 14336
    d = glu_synth.gemm_llama(M=M, K=K, I=I, dtype="bf16", exact=exact)
    xd, gd, ud = (to_dev(d[k], "bf16") for k in ("x", "w_gate", "w_up"))
    y = glu.gemm_fwd(xd, gd, ud, act="silu")
    torch.cuda.synchronize()
    ms, is_ = sample_positions(M, I, 4096, 16)
    yb = to_bits(y, "bf16")[ms, is_]
    ref, g, u, sg, su = orc.gemm_glu_at("silu", "bf16", d["x"], d["w_gate"], d["w_up"], ms, is_)
    if exact:
        compare(yb, ref, "bf16", what="full layer grid")
    else:
        check_bound(orc, "silu", "bf16", yb, g, u, sg, su, K, "full layer normal")
    assert not torch.isnan(y).any()


def test_host_memory_operands_are_refused():
    """The tensor-memory accelerator path takes device memory only: a pinned
    host operand is refused before any launch (GLU_ERR_VALUE)."""
    x = torch.zeros(128, 64, dtype=torch.bfloat16).pin_memory()
    w = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(128, 64, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = glu.glu_gemm_fwd(x.data_ptr(), 64, w.data_ptr(), w.data_ptr(), 64, y.data_ptr(), 64, 128, 64, 64, 0, 2, s)
    assert st == -8
    yh = torch.zeros(128, 64, dtype=torch.bfloat16).pin_memory()
    xd = x.cuda()
    st = glu.glu_gemm_fwd(xd.data_ptr(), 64, w.data_ptr(), w.data_ptr(), 64, yh.data_ptr(), 64, 128, 64, 64, 0, 2, s)
    assert st == -8
