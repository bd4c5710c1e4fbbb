"""The host-memory entry points (glu_fwd_host, glu_bwd_host) against the
oracle: blocks of rows streamed through a small device workspace, so that a
call runs many blocks with a ragged last one, on page-locked and pageable
memory, strided and [gate | up] layouts, in place, and with one stream or
three."""
import numpy as np
import pytest
import torch

import glu_activation_mlps_gb300 as glu
import glu_synth
import helpers
from helpers import compare

pytestmark = pytest.mark.gpu

NP_SIGNED = {"f32": np.int32, "f16": np.int16, "bf16": np.int16}
TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
BITS = {"f32": np.uint32, "f16": np.uint16, "bf16": np.uint16}


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    glu.build()
    glu.lib()
    glu.glu_set_tuning(0, 0, 0, 0)


def host(bits, dt, pinned=True):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(NP_SIGNED[dt])).view(TORCH[dt])
    return t.pin_memory() if pinned else t.clone()


def bits_of(t, dt):
    return t.contiguous().view({"f32": torch.int32, "f16": torch.int16, "bf16": torch.int16}[dt]).numpy().view(BITS[dt])


def pipe_for(rows_per_block, cols, layout, dt, backward):
    need = glu.glu_host_workspace_bytes(rows_per_block, cols, glu.LAYOUT[layout], glu.DTYPE[dt], backward)
    return glu.HostPipeline(workspace_bytes=need)


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("pinned", [True, False])
def test_host_split(orc, dt, pinned):
    rows, cols = 301, 1000
    rng = np.random.default_rng(7)
    a = glu_synth.normal_bits(rng, (rows, cols), 2.0, dt)
    b = glu_synth.normal_bits(rng, (rows, cols), 1.0, dt)
    dc = glu_synth.normal_bits(rng, (rows, cols), 1.0, dt)
    for act in ("silu", "gelu_erf"):
        p = pipe_for(37, cols, "split", dt, 1)              # 9 blocks, the last one of 5 rows
        A, B, DC = host(a, dt, pinned), host(b, dt, pinned), host(dc, dt, pinned)
        y = glu.fwd_host(p, A, B, act=act)
        da, db = glu.bwd_host(p, DC, A, B, act=act)
        torch.cuda.current_stream().synchronize()
        compare(bits_of(y, dt), orc.fwd(act, dt, a, b), dt, what=f"{act} {dt} host fwd")
        scale = orc.bwd_da_scale(act, dt, dc, a, b) if dt == "f32" else None
        da_o, db_o = orc.bwd(act, dt, dc, a, b)
        compare(bits_of(da, dt), da_o, dt, scale=scale, what=f"{act} {dt} host da")
        compare(bits_of(db, dt), db_o, dt, what=f"{act} {dt} host db")


def test_host_strided_concat_and_inplace(orc):
    dt, rows, cols = "bf16", 129, 777
    rng = np.random.default_rng(8)
    x = glu_synth.normal_bits(rng, (rows, 2 * cols), 1.5, dt)
    dc = glu_synth.normal_bits(rng, (rows, cols), 1.0, dt)
    # x inside a wider pinned buffer: row stride 2*cols + 9
    buf = torch.zeros((rows, 2 * cols + 9), dtype=torch.bfloat16).pin_memory()
    X = buf[:, :2 * cols]
    X.copy_(host(x, dt))
    p = pipe_for(16, cols, "concat", dt, 1)
    y = glu.fwd_host(p, X, layout="concat", act="gelu_tanh")
    torch.cuda.current_stream().synchronize()
    y_o = orc.fwd_concat("gelu_tanh", dt, x, cols)
    compare(bits_of(y, dt), y_o, dt, what="host concat fwd")
    dx = glu.bwd_host(p, host(dc, dt), X, layout="concat", act="gelu_tanh")
    torch.cuda.current_stream().synchronize()
    dx_o = orc.bwd_concat("gelu_tanh", dt, dc, x, cols)
    compare(bits_of(dx, dt)[:, :cols], dx_o[:, :cols], dt, what="host concat da")
    compare(bits_of(dx, dt)[:, cols:], dx_o[:, cols:], dt, what="host concat db")
    # in place over the up half of x, on the host
    glu.fwd_host(p, X, layout="concat", y=X[:, cols:], act="gelu_tanh")
    torch.cuda.current_stream().synchronize()
    compare(bits_of(X[:, cols:], dt), y_o, dt, what="host concat in place")
    assert np.array_equal(bits_of(X[:, :cols], dt), x[:, :cols])
    assert (bits_of(buf[:, 2 * cols:], dt) == 0).all()       # padding untouched


def test_host_single_stream_and_inplace_backward(orc):
    dt, rows, cols = "f16", 200, 2048
    rng = np.random.default_rng(9)
    a = glu_synth.normal_bits(rng, (rows, cols), 2.0, dt)
    b = glu_synth.normal_bits(rng, (rows, cols), 1.0, dt)
    dc = glu_synth.normal_bits(rng, (rows, cols), 1.0, dt)
    need = glu.glu_host_workspace_bytes(30, cols, 0, glu.DTYPE[dt], 1)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    A, B, DC = host(a, dt), host(b, dt), host(dc, dt)
    st = glu.glu_bwd_host(DC.data_ptr(), cols, A.data_ptr(), cols, B.data_ptr(), cols, A.data_ptr(), cols,
                          B.data_ptr(), cols, rows, cols, 0, 0, glu.DTYPE[dt], ws.data_ptr(), need, s, s, s)
    assert st == 0
    torch.cuda.current_stream().synchronize()
    da_o, db_o = orc.bwd("silu", dt, dc, a, b)
    compare(bits_of(A, dt), da_o, dt, what="host in-place da")
    compare(bits_of(B, dt), db_o, dt, what="host in-place db")


def test_host_metric_workload_sampled(orc):
    d = glu_synth.metric_bf16()
    A, B, DC = host(d["a"], "bf16"), host(d["b"], "bf16"), host(d["dc"], "bf16")
    p = glu.HostPipeline(workspace_bytes=256 << 20)
    y = glu.fwd_host(p, A, B)
    da, db = glu.bwd_host(p, DC, A, B)
    torch.cuda.current_stream().synchronize()
    rng = np.random.default_rng(1)
    idx = rng.integers(0, d["a"].size, 1 << 18)
    a_s, b_s, dc_s = (d[k].ravel()[idx] for k in ("a", "b", "dc"))
    compare(bits_of(y, "bf16").ravel()[idx], orc.fwd("silu", "bf16", a_s, b_s), "bf16", what="metric host y")
    da_o, db_o = orc.bwd("silu", "bf16", dc_s, a_s, b_s)
    compare(bits_of(da, "bf16").ravel()[idx], da_o, "bf16", what="metric host da")
    compare(bits_of(db, "bf16").ravel()[idx], db_o, "bf16", what="metric host db")


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_device_entry_points_on_pinned_host_memory(orc, dt):
    """glu_fwd / glu_bwd on pinned host buffers (the kernels read and write them
    in place over the host link): element by element against the oracle."""
    rows, cols = 300, 2000
    rng = np.random.default_rng(77)
    a = glu_synth.normal_bits(rng, (rows, cols), 2.0, dt)
    b = glu_synth.normal_bits(rng, (rows, cols), 1.0, dt)
    dc = glu_synth.normal_bits(rng, (rows, cols), 1.0, dt)
    T = helpers.TORCH[dt]
    pin = lambda bits: torch.from_numpy(bits.view(helpers.NP_SIGNED[dt])).view(T).pin_memory()
    A, B, DC = pin(a), pin(b), pin(dc)
    Y, DA, DB = (torch.empty(rows, cols, dtype=T).pin_memory() for _ in range(3))
    s = torch.cuda.current_stream().cuda_stream
    code = {"bf16": 2, "f32": 0}[dt]
    assert glu.glu_fwd(A.data_ptr(), cols, B.data_ptr(), cols, Y.data_ptr(), cols, rows, cols, 0, 0, code, s) == 0
    assert glu.glu_bwd(DC.data_ptr(), cols, A.data_ptr(), cols, B.data_ptr(), cols, DA.data_ptr(), cols,
                       DB.data_ptr(), cols, rows, cols, 0, 0, code, s) == 0
    torch.cuda.synchronize()
    bits = lambda t: t.view(helpers.TORCH_INT[dt]).numpy().view(helpers.NP_BITS[dt])
    helpers.compare(bits(Y), orc.fwd("silu", dt, a, b), dt, what="zero-copy y")
    da, db = orc.bwd("silu", dt, dc, a, b)
    scale = orc.bwd_da_scale("silu", dt, dc, a, b) if dt == "f32" else None
    helpers.compare(bits(DA), da, dt, scale=scale, what="zero-copy da")
    helpers.compare(bits(DB), db, dt, what="zero-copy db")


def test_bulk_path_leaves_pinned_host_inputs_to_direct_loads(orc):
    """With the bulk-copy path selected, inputs in pinned host memory still take
    the direct kernels (the bulk-copy engine is given device memory only), and
    the results are the oracle's."""
    rows, cols, dt = 300, 2000, "bf16"
    rng = np.random.default_rng(78)
    a = glu_synth.normal_bits(rng, (rows, cols), 2.0, dt)
    b = glu_synth.normal_bits(rng, (rows, cols), 1.0, dt)
    T = helpers.TORCH[dt]
    pin = lambda bits: torch.from_numpy(bits.view(helpers.NP_SIGNED[dt])).view(T).pin_memory()
    A, B = pin(a), pin(b)
    Y = torch.empty(rows, cols, dtype=T).pin_memory()
    s = torch.cuda.current_stream().cuda_stream
    glu.glu_set_tuning(0, 0, 0, 0, 2)
    try:
        assert glu.glu_fwd(A.data_ptr(), cols, B.data_ptr(), cols, Y.data_ptr(), cols, rows, cols, 0, 0, 2, s) == 0
        torch.cuda.synchronize()
        assert glu.glu_last_launch()["path"] == 1
        # the same call on device copies does take the bulk path
        Ad, Bd, Yd = A.cuda(), B.cuda(), torch.empty(rows, cols, dtype=T, device="cuda")
        assert glu.glu_fwd(Ad.data_ptr(), cols, Bd.data_ptr(), cols, Yd.data_ptr(), cols, rows, cols, 0, 0, 2, s) == 0
        torch.cuda.synchronize()
        assert glu.glu_last_launch()["path"] == 2
    finally:
        glu.glu_set_tuning(0, 0, 0, 0, 0)
    bits = lambda t: t.view(helpers.TORCH_INT[dt]).cpu().numpy().view(helpers.NP_BITS[dt])
    y = orc.fwd("silu", dt, a, b)
    helpers.compare(bits(Y), y, dt, what="pinned inputs, bulk path selected")
    helpers.compare(bits(Yd), y, dt, what="device inputs, bulk path")
