"""GPU parity: the CUDA library against the double-precision oracle on the same
seeded inputs, element by element.

Small cases cover every activation x dtype x direction on shapes that span
several tiles with ragged tails, strided rows, the [gate | up] layout, the
in-place variants and misaligned bases.  The named workloads run at full size
in the launch configuration the benchmark times; the oracle checks every
element where it finishes in seconds and a seeded sample otherwise."""
import os

import numpy as np
import pytest
import torch

import glu_activation_mlps_gb300 as glu
import glu_synth
from helpers import compare, to_bits, to_dev

pytestmark = pytest.mark.gpu

ACTS = ("silu", "gelu_erf", "gelu_tanh", "relu")
DTYPES = ("bf16", "f16", "f32")
THREADS = max(1, min(32, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    glu.build()
    glu.lib()
    glu.glu_set_tuning(0, 0, 0)


def oracle_check_fwd(orc, act, dt, a, b, y_gpu, what):
    y = orc.fwd_threaded(act, dt, a, b, THREADS)
    return compare(y_gpu, y, dt, what=what)


def oracle_check_bwd(orc, act, dt, dc, a, b, da_gpu, db_gpu, what):
    da, db = orc.bwd_threaded(act, dt, dc, a, b, THREADS)
    scale = orc.bwd_da_scale(act, dt, dc, a, b) if dt == "f32" else None
    s1 = compare(da_gpu, da, dt, scale=scale, what=what + " da")
    s2 = compare(db_gpu, db, dt, what=what + " db")
    return s1, s2


def inputs(shape, dt, seed, sigma_a=2.5):
    rng = np.random.default_rng(seed)
    a = glu_synth.normal_bits(rng, shape, sigma_a, dt)
    b = glu_synth.normal_bits(rng, shape, 1.0, dt)
    dc = glu_synth.normal_bits(rng, shape, 1.0, dt)
    return a, b, dc


# ---------------------------------------------------------------- small shapes

SHAPES = [(1, 1), (1, 7), (3, 17), (64, 1000), (33, 3001), (5, 16385)]


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("act", ACTS)
def test_contiguous_shapes(orc, act, dt):
    for i, shape in enumerate(SHAPES):
        a, b, dc = inputs(shape, dt, 100 + i)
        A, B, DC = to_dev(a, dt), to_dev(b, dt), to_dev(dc, dt)
        y = glu.fwd(A, B, act=act)
        oracle_check_fwd(orc, act, dt, a, b, to_bits(y, dt), f"{act} {dt} {shape} fwd")
        da, db = glu.bwd(DC, A, B, act=act)
        oracle_check_bwd(orc, act, dt, dc, a, b, to_bits(da, dt), to_bits(db, dt), f"{act} {dt} {shape} bwd")


def strided(base_shape_cols, rows, cols, dt, bits):
    """A (rows, cols) view with row stride base_shape_cols, holding `bits`."""
    buf = torch.zeros((rows, base_shape_cols), dtype=torch.int32 if dt == "f32" else torch.int16, device="cuda")
    buf = buf.view({"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dt])
    v = buf[:, :cols]
    v.copy_(to_dev(bits, dt))
    return v


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("act", ACTS)
def test_strided_rows(orc, act, dt):
    """Rows with per-operand strides: the row path (not flattened), both with
    aligned strides (vector units + a one-element tail) and unaligned ones."""
    # first case: every stride a multiple of 16 elements (32-byte aligned rows);
    # second case: odd strides, so only element-wide accesses are possible
    for rows, cols, pads in ((9, 4001, (15, 47, 31, 63, 79, 95)), (6, 1029, (1, 3, 5, 7, 9, 11))):
        a, b, dc = inputs((rows, cols), dt, 7 + cols)
        A = strided(cols + pads[0], rows, cols, dt, a)
        B = strided(cols + pads[1], rows, cols, dt, b)
        DC = strided(cols + pads[2], rows, cols, dt, dc)
        Y = strided(cols + pads[3], rows, cols, dt, np.zeros_like(a))
        glu.fwd(A, B, y=Y, act=act)
        info = glu.glu_last_launch()
        assert info["launched"] == 1 and info["flattened"] == 0
        if pads[0] == 15:
            assert info["vec_bytes"] >= 16 and info["tail_elems"] == rows
        oracle_check_fwd(orc, act, dt, a, b, to_bits(Y, dt), f"{act} {dt} strided fwd")
        DA = strided(cols + pads[4], rows, cols, dt, np.zeros_like(a))
        DB = strided(cols + pads[5], rows, cols, dt, np.zeros_like(a))
        glu.bwd(DC, A, B, da=DA, db=DB, act=act)
        oracle_check_bwd(orc, act, dt, dc, a, b, to_bits(DA, dt), to_bits(DB, dt), f"{act} {dt} strided bwd")


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("act", ACTS)
def test_concat_layout_and_inplace(orc, act, dt):
    for rows, cols in ((12, 1280), (7, 1234), (3, 5)):
        rng = np.random.default_rng(cols)
        x = glu_synth.normal_bits(rng, (rows, 2 * cols), 2.0, dt)
        dc = glu_synth.normal_bits(rng, (rows, cols), 1.0, dt)
        X = to_dev(x, dt)
        y = glu.fwd(X, layout="concat", act=act)
        y_or = orc.fwd_concat(act, dt, x, cols)
        compare(to_bits(y, dt), y_or, dt, what=f"{act} {dt} concat fwd")
        # in place over the up half: y = x[:, I:]
        X2 = to_dev(x, dt)
        glu.fwd(X2, layout="concat", y=X2[:, cols:], act=act)
        compare(to_bits(X2[:, cols:], dt), y_or, dt, what=f"{act} {dt} concat fwd in place")
        assert np.array_equal(to_bits(X2[:, :cols], dt), x[:, :cols])       # gate half untouched
        # backward: dx = [da | db], out of place and over x
        DC = to_dev(dc, dt)
        dx = glu.bwd(DC, X, layout="concat", act=act)
        dx_or = orc.bwd_concat(act, dt, dc, x, cols)
        a, b = x[:, :cols], x[:, cols:]
        scale = orc.bwd_da_scale(act, dt, dc, a, b) if dt == "f32" else None
        compare(to_bits(dx, dt)[:, :cols], dx_or[:, :cols], dt, scale=scale, what=f"{act} {dt} concat da")
        compare(to_bits(dx, dt)[:, cols:], dx_or[:, cols:], dt, what=f"{act} {dt} concat db")
        X3 = to_dev(x, dt)
        glu.bwd(DC, X3, layout="concat", inplace=True, act=act)
        got = to_bits(X3, dt)
        compare(got[:, :cols], dx_or[:, :cols], dt, scale=scale, what=f"{act} {dt} concat da in place")
        compare(got[:, cols:], dx_or[:, cols:], dt, what=f"{act} {dt} concat db in place")


@pytest.mark.parametrize("dt", DTYPES)
def test_split_inplace(orc, dt):
    for act in ACTS:
        a, b, dc = inputs((37, 2050), dt, 3)
        A, B, DC = to_dev(a, dt), to_dev(b, dt), to_dev(dc, dt)
        glu.fwd(A, B, y=B, act=act)                                   # y over b
        oracle_check_fwd(orc, act, dt, a, b, to_bits(B, dt), f"{act} {dt} fwd over b")
        assert np.array_equal(to_bits(A, dt), a)
        A, B = to_dev(a, dt), to_dev(b, dt)
        glu.bwd(DC, A, B, inplace=True, act=act)                      # da over a, db over b
        oracle_check_bwd(orc, act, dt, dc, a, b, to_bits(A, dt), to_bits(B, dt), f"{act} {dt} bwd in place")
        assert np.array_equal(to_bits(DC, dt), dc)


@pytest.mark.parametrize("dt", DTYPES)
def test_misaligned_bases_use_element_accesses(orc, dt):
    E = 4 if dt == "f32" else 2
    n = 4099
    a, b, dc = inputs((n,), dt, 21)
    for off in (1, 3):
        bufs = [torch.empty(n + 8, dtype={"f32": torch.float32, "f16": torch.float16,
                                         "bf16": torch.bfloat16}[dt], device="cuda") for _ in range(3)]
        A, B, Y = (t[off:off + n] for t in bufs)
        A.copy_(to_dev(a, dt))
        B.copy_(to_dev(b, dt))
        glu.fwd(A, B, y=Y, act="silu")
        info = glu.glu_last_launch()
        assert info["vec_bytes"] == E and info["tail_elems"] == n
        oracle_check_fwd(orc, "silu", dt, a, b, to_bits(Y, dt), f"{dt} misaligned {off}")


def test_stream_argument_is_honoured(orc):
    a, b, _ = inputs((256, 4096), "bf16", 5)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        A, B = to_dev(a, "bf16"), to_dev(b, "bf16")
        y = glu.fwd(A, B, act="silu", stream=s)
    s.synchronize()
    oracle_check_fwd(orc, "silu", "bf16", a, b, to_bits(y, "bf16"), "side stream")


# ---------------------------------------------------------------- named workloads at full size

def test_fwd_f32_256x1024(orc):
    d = glu_synth.fwd_f32_small()
    A, B = to_dev(d["a"], "f32"), to_dev(d["b"], "f32")
    y = glu.fwd(A, B, act="silu")
    info = glu.glu_last_launch()
    assert info["vec_bytes"] == 32 and info["flattened"] == 1 and info["tail_elems"] == 0
    st = oracle_check_fwd(orc, "silu", "f32", d["a"], d["b"], to_bits(y, "f32"), "fwd f32 256x1024")
    assert st["max_plain_rel"] < 1e-6                 # plain relative error holds for the forward


def test_fwd_bf16_4096x11008(orc):
    d = glu_synth.fwd_bf16_split()
    A, B = to_dev(d["a"], "bf16"), to_dev(d["b"], "bf16")
    y = glu.fwd(A, B, act="silu")
    info = glu.glu_last_launch()
    assert info["vec_bytes"] == 32 and info["flattened"] == 1
    oracle_check_fwd(orc, "silu", "bf16", d["a"], d["b"], to_bits(y, "bf16"), "fwd bf16 4096x11008")


def test_fwd_bf16_concat_4096x18944(orc):
    d = glu_synth.fwd_bf16_concat()
    x, C = d["x"], d["n_cols"]
    y_or = orc.fwd_threaded("silu", "bf16", np.ascontiguousarray(x[:, :C]), np.ascontiguousarray(x[:, C:]),
                            THREADS)
    X = to_dev(x, "bf16")
    y = glu.fwd(X, layout="concat", act="silu")
    info = glu.glu_last_launch()
    assert info["vec_bytes"] == 32 and info["flattened"] == 0 and info["tail_elems"] == 0
    compare(to_bits(y, "bf16"), y_or, "bf16", what="concat out of place")
    glu.fwd(X, layout="concat", y=X[:, C:], act="silu")
    got = to_bits(X, "bf16")
    compare(got[:, C:], y_or, "bf16", what="concat in place over b")
    assert np.array_equal(got[:, :C], x[:, :C])


def test_bwd_bf16_4096x28672_inplace_with_outliers(orc):
    d = glu_synth.bwd_bf16_outliers()
    A, B, DC = to_dev(d["a"], "bf16"), to_dev(d["b"], "bf16"), to_dev(d["dc"], "bf16")
    glu.bwd(DC, A, B, inplace=True, act="silu")
    info = glu.glu_last_launch()
    assert info["backward"] == 1 and info["vec_bytes"] >= 16 and info["flattened"] == 1
    oracle_check_bwd(orc, "silu", "bf16", d["dc"], d["a"], d["b"], to_bits(A, "bf16"), to_bits(B, "bf16"),
                     "bwd bf16 4096x28672 in place")
    a_vals = orc.decode("bf16", d["a"])
    assert np.isin([-88.0, 88.0], a_vals).all()      # the outliers are present


def test_metric_workload_fwd_bwd(orc):
    d = glu_synth.metric_bf16()
    A, B, DC = to_dev(d["a"], "bf16"), to_dev(d["b"], "bf16"), to_dev(d["dc"], "bf16")
    y = glu.fwd(A, B, act="silu")
    da, db = glu.bwd(DC, A, B, act="silu")
    oracle_check_fwd(orc, "silu", "bf16", d["a"], d["b"], to_bits(y, "bf16"), "metric fwd")
    oracle_check_bwd(orc, "silu", "bf16", d["dc"], d["a"], d["b"], to_bits(da, "bf16"), to_bits(db, "bf16"),
                     "metric bwd")


def sampled(rows, cols, k, seed):
    rng = np.random.default_rng(seed)
    idx = rng.integers(0, rows * cols, size=k)
    edges = np.concatenate([np.arange(cols), (rows - 1) * cols + np.arange(cols)])
    return np.unique(np.concatenate([idx, edges]))


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("H", glu_synth.SWEEP_H)
def test_activation_sweep_full_size(orc, H, dt):
    """4096 x H, every activation, forward and backward, on the full tensors;
    the oracle checks a seeded sample plus the first and last rows."""
    d = glu_synth.sweep(H, dt)
    A, B, DC = to_dev(d["a"], dt), to_dev(d["b"], dt), to_dev(d["dc"], dt)
    idx = sampled(4096, H, 1 << 17, H)
    a_s, b_s, dc_s = d["a"].ravel()[idx], d["b"].ravel()[idx], d["dc"].ravel()[idx]
    idx_t = torch.from_numpy(idx).cuda()
    for act in ACTS:
        y = glu.fwd(A, B, act=act)
        assert glu.glu_last_launch()["vec_bytes"] >= 16
        compare(to_bits(y.view(-1)[idx_t], dt), orc.fwd(act, dt, a_s, b_s), dt, what=f"{act} {dt} H={H} fwd")
        da, db = glu.bwd(DC, A, B, act=act)
        scale = orc.bwd_da_scale(act, dt, dc_s, a_s, b_s) if dt == "f32" else None
        da_o, db_o = orc.bwd(act, dt, dc_s, a_s, b_s)
        compare(to_bits(da.view(-1)[idx_t], dt), da_o, dt, scale=scale, what=f"{act} {dt} H={H} da")
        compare(to_bits(db.view(-1)[idx_t], dt), db_o, dt, what=f"{act} {dt} H={H} db")


# ---------------------------------------------------------------- dependent launches

@pytest.mark.parametrize("dependent", [0, -1])
def test_back_to_back_dependent_kernels(orc, dependent):
    """A chain of launches on one stream in which every launch reads what the
    previous one wrote (forward output -> next forward's gate, backward inputs
    from the chain).  Values are signed powers of two and the activation is
    ReLU, so every product is exact: the GPU chain must equal the oracle's
    chain bit for bit, and any launch that read its input before the previous
    kernel finished writing it would show up as a mismatch.  Run with and
    without programmatic dependent launch.  The launches (34-50 MB of inputs)
    also prefetch their first tile into L2 before waiting on the previous
    launch, which this chain checks cannot expose data older than its writes."""
    glu.glu_set_tuning(0, 0, 0, dependent)
    try:
        rows, cols, dt = 2048, 4096, "bf16"
        rng = np.random.default_rng(99)
        pick = np.array([-2.0, -1.0, -0.5, 0.5, 1.0, 2.0])
        a = orc.encode(dt, rng.choice(pick, (rows, cols)))
        b = orc.encode(dt, rng.choice(pick, (rows, cols)))
        x_gpu, B = to_dev(a, dt), to_dev(b, dt)
        x_orc = a
        n = 40
        # every output buffer starts as NaN and is allocated before the chain,
        # so that only the library's kernels run back to back on the stream
        bufs = [torch.full_like(x_gpu, float("nan")) for _ in range(n + n // 4)]
        torch.cuda.synchronize()
        outs = []
        for k in range(n):
            if k % 4 == 3:      # backward: dc = x, a = x  ->  da, db feed the chain
                da, db = bufs.pop(), bufs.pop()
                glu.bwd(x_gpu, x_gpu, B, da=da, db=db, act="relu")
                da_o, db_o = orc.bwd("relu", dt, x_orc, x_orc, b)
                x_gpu, x_orc = db, db_o
                outs.append((da, da_o))
            else:
                y = bufs.pop()
                glu.fwd(x_gpu, B, y=y, act="relu")
                x_orc = orc.fwd("relu", dt, x_orc, b)
                x_gpu = y
        torch.cuda.synchronize()
        assert np.array_equal(to_bits(x_gpu, dt), x_orc)
        for g, o in outs:
            assert np.array_equal(to_bits(g, dt), o)
    finally:
        glu.glu_set_tuning(0, 0, 0, 0)
