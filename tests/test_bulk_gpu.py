"""The bulk-copy staging path (glu_tuning_t.path = 2) against the oracle:
contiguous operands whose whole 16 KiB chunks are staged in shared memory by
the bulk-copy engine, with the remainder on the direct path; small inputs and
misaligned bases fall back to the direct path.  Guard bands check that no
byte outside an output is written, and the device counter of waits that ran
out must stay at zero."""
import numpy as np
import pytest
import torch

import glu_activation_mlps_gb300 as glu
import glu_synth
from helpers import compare, to_bits, to_dev

pytestmark = pytest.mark.gpu

ACTS = ("silu", "gelu_erf", "gelu_tanh", "relu")


@pytest.fixture(scope="module", autouse=True, params=[0, 1], ids=["narrow", "wide"])
def bulk_path(request):
    """ctas_per_sm 1 selects the one-block-per-SM shape, 0 the two-block one."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    glu.build()
    glu.lib()
    glu.glu_wait_timeouts(reset=True)
    glu.glu_set_tuning(0, 0, request.param, 0, 2)
    yield
    glu.glu_set_tuning(0, 0, 0, 0, 0)


def check_case(orc, act, dt, shape, seed, expect_bulk):
    rng = np.random.default_rng(seed)
    a = glu_synth.normal_bits(rng, shape, 2.0, dt)
    b = glu_synth.normal_bits(rng, shape, 1.0, dt)
    dc = glu_synth.normal_bits(rng, shape, 1.0, dt)
    A, B, DC = to_dev(a, dt), to_dev(b, dt), to_dev(dc, dt)
    y = glu.fwd(A, B, act=act)
    assert glu.glu_last_launch()["path"] == (2 if expect_bulk else 1)
    compare(to_bits(y, dt), orc.fwd(act, dt, a, b), dt, what=f"bulk {act} {dt} {shape} fwd")
    da, db = glu.bwd(DC, A, B, act=act)
    assert glu.glu_last_launch()["path"] == (2 if expect_bulk else 1)
    scale = orc.bwd_da_scale(act, dt, dc, a, b) if dt == "f32" else None
    da_o, db_o = orc.bwd(act, dt, dc, a, b)
    compare(to_bits(da, dt), da_o, dt, scale=scale, what=f"bulk {act} {dt} {shape} da")
    compare(to_bits(db, dt), db_o, dt, what=f"bulk {act} {dt} {shape} db")


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("act", ACTS)
def test_bulk_matches_oracle(orc, act, dt):
    check_case(orc, act, dt, (64, 1000), 1, True)          # whole chunks plus a remainder
    check_case(orc, act, dt, (512, 2048), 2, True)         # exact chunks, several per block
    check_case(orc, act, dt, (3, 17), 3, False)            # below one chunk: direct path


def test_bulk_inplace_and_guard_bands(orc):
    dt = "bf16"
    n = 3 * 8192 + 77                                      # 3 chunks of 8192 bf16 + a remainder
    rng = np.random.default_rng(5)
    a = glu_synth.normal_bits(rng, (n,), 2.0, dt)
    b = glu_synth.normal_bits(rng, (n,), 1.0, dt)
    dc = glu_synth.normal_bits(rng, (n,), 1.0, dt)
    guard = 4096
    buf = torch.full((n + 2 * guard,), 0x7FAD, dtype=torch.int16, device="cuda")
    Y = buf[guard:guard + n].view(torch.bfloat16)
    glu.fwd(to_dev(a, dt), to_dev(b, dt), y=Y, act="silu")
    assert glu.glu_last_launch()["path"] == 2
    host = buf.cpu().numpy().view(np.uint16)
    assert (host[:guard] == 0x7FAD).all() and (host[guard + n:] == 0x7FAD).all()
    compare(to_bits(Y, dt), orc.fwd("silu", dt, a, b), dt, what="bulk guarded")
    # in place: y over b, and da over a, db over b
    A, B, DC = to_dev(a, dt), to_dev(b, dt), to_dev(dc, dt)
    glu.fwd(A, B, y=B, act="gelu_tanh")
    compare(to_bits(B, dt), orc.fwd("gelu_tanh", dt, a, b), dt, what="bulk fwd over b")
    A, B = to_dev(a, dt), to_dev(b, dt)
    glu.bwd(DC, A, B, inplace=True, act="gelu_tanh")
    da_o, db_o = orc.bwd("gelu_tanh", dt, dc, a, b)
    compare(to_bits(A, dt), da_o, dt, what="bulk da over a")
    compare(to_bits(B, dt), db_o, dt, what="bulk db over b")


def test_bulk_misaligned_base_falls_back(orc):
    dt = "f16"
    n = 40000
    rng = np.random.default_rng(6)
    a = glu_synth.normal_bits(rng, (n,), 2.0, dt)
    b = glu_synth.normal_bits(rng, (n,), 1.0, dt)
    bufs = [torch.empty(n + 8, dtype=torch.float16, device="cuda") for _ in range(3)]
    A, B, Y = (t[1:1 + n] for t in bufs)
    A.copy_(to_dev(a, dt))
    B.copy_(to_dev(b, dt))
    glu.fwd(A, B, y=Y, act="relu")
    assert glu.glu_last_launch()["path"] == 1
    compare(to_bits(Y, dt), orc.fwd("relu", dt, a, b), dt, what="bulk fallback")


def test_bulk_metric_workload_sampled(orc):
    d = glu_synth.metric_bf16()
    A, B, DC = to_dev(d["a"], "bf16"), to_dev(d["b"], "bf16"), to_dev(d["dc"], "bf16")
    y = glu.fwd(A, B)
    da, db = glu.bwd(DC, A, B)
    assert glu.glu_last_launch()["path"] == 2
    idx = np.random.default_rng(3).integers(0, d["a"].size, 1 << 18)
    a_s, b_s, dc_s = (d[k].ravel()[idx] for k in ("a", "b", "dc"))
    t = torch.from_numpy(idx).cuda()
    compare(to_bits(y.view(-1)[t], "bf16"), orc.fwd("silu", "bf16", a_s, b_s), "bf16", what="bulk metric y")
    da_o, db_o = orc.bwd("silu", "bf16", dc_s, a_s, b_s)
    compare(to_bits(da.view(-1)[t], "bf16"), da_o, "bf16", what="bulk metric da")
    compare(to_bits(db.view(-1)[t], "bf16"), db_o, "bf16", what="bulk metric db")


def test_no_wait_ran_out():
    torch.cuda.synchronize()
    assert glu.glu_wait_timeouts() == 0
