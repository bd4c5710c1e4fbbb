"""Brute force over the whole input domain of the activation: every finite
bf16 and f16 value of a, with b and dc fixed to a few values, forward and
backward, all activations, against the oracle under the 1-ulp bar.  For f32,
a dense sweep of a over [-200, 80], denser still around the derivative roots
and in the tails, under the fp32 bar.
Non-finite and extreme inputs only have to run without faulting and keep
their sign/NaN behaviour."""
import numpy as np
import pytest
import torch

import glu_activation_mlps_gb300 as glu
import glu_synth
from helpers import compare, to_bits, to_dev

pytestmark = pytest.mark.gpu

ACTS = ("silu", "gelu_erf", "gelu_tanh", "relu")
B_VALUES = (1.0, -3.5, 0.0078125, 100.0)
DC_VALUES = (1.0, 0.75)


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    glu.build()
    glu.lib()
    glu.glu_set_tuning(0, 0, 0)


def const_bits(orc, dt, v, n):
    return np.full(n, orc.encode(dt, [v])[0], dtype=orc.BITS_DTYPE[dt])


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("act", ACTS)
def test_every_16bit_input(orc, act, dt):
    a = glu_synth.all_finite_16bit(dt)
    n = a.size
    A = to_dev(a, dt)
    worst = {}
    for bv in B_VALUES:
        b = const_bits(orc, dt, bv, n)
        B = to_dev(b, dt)
        y = glu.fwd(A, B, act=act)
        worst[("fwd", bv)] = compare(to_bits(y, dt), orc.fwd(act, dt, a, b), dt, what=f"{act} {dt} b={bv}")
        for cv in DC_VALUES:
            dc = const_bits(orc, dt, cv, n)
            da, db = glu.bwd(to_dev(dc, dt), A, B, act=act)
            da_o, db_o = orc.bwd(act, dt, dc, a, b)
            worst[("da", bv, cv)] = compare(to_bits(da, dt), da_o, dt, what=f"{act} {dt} da b={bv} dc={cv}")
            worst[("db", bv, cv)] = compare(to_bits(db, dt), db_o, dt, what=f"{act} {dt} db b={bv} dc={cv}")
    assert all(s["max_ulp"] <= 1 for s in worst.values())


def f32_grid():
    rng = np.random.default_rng(77)
    parts = [
        np.linspace(-200, 80, 600001),
        rng.uniform(-8, 8, 400000),
        rng.uniform(-16, -6, 200000),                               # GELU tails
        -1.2784645427610738 + np.linspace(-1e-2, 1e-2, 20001),     # silu' root
        -0.7517915246935645 + np.linspace(-1e-2, 1e-2, 20001),     # gelu-erf' root
        -0.7524614220710163 + np.linspace(-1e-2, 1e-2, 20001),     # gelu-tanh' root
        np.geomspace(1e-30, 80, 20000), -np.geomspace(1e-30, 200, 20000),
    ]
    return np.concatenate(parts).astype(np.float32).view(np.uint32)


@pytest.mark.parametrize("act", ACTS)
def test_dense_f32_sweep(orc, act):
    """f32 a over [-200, 80] (deep tails included: there the fp32 bar's
    absolute floor applies), denser near the derivative roots."""
    a = f32_grid()
    n = a.size
    A = to_dev(a, "f32")
    for bv in (1.0, -3.5):
        b = const_bits(orc, "f32", bv, n)
        B = to_dev(b, "f32")
        y = glu.fwd(A, B, act=act)
        st = compare(to_bits(y, "f32"), orc.fwd(act, "f32", a, b), "f32", what=f"{act} f32 fwd b={bv}")
        for cv in (1.0, 0.75):
            dc = const_bits(orc, "f32", cv, n)
            da, db = glu.bwd(to_dev(dc, "f32"), A, B, act=act)
            da_o, db_o = orc.bwd(act, "f32", dc, a, b)
            scale = orc.bwd_da_scale(act, "f32", dc, a, b)
            compare(to_bits(da, "f32"), da_o, "f32", scale=scale, what=f"{act} f32 da b={bv}")
            compare(to_bits(db, "f32"), db_o, "f32", what=f"{act} f32 db b={bv}")
            v = to_bits(da, "f32").view(np.float32)
            assert np.isfinite(v).all()


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
def test_non_finite_and_extreme_inputs_do_not_fault(orc, dt):
    vals = [float("nan"), float("inf"), -float("inf"), 3.0e38 if dt != "f16" else 65504.0,
            -3.0e38 if dt != "f16" else -65504.0, 0.0, -0.0, -1.0e4, 1.0e4]
    a = orc.encode(dt, np.array(vals))
    b = orc.encode(dt, np.ones(len(vals)))
    A, B = to_dev(a, dt), to_dev(b, dt)
    for act in ACTS:
        y = to_bits(glu.fwd(A, B, act=act), dt)
        da, db = glu.bwd(B, A, B, act=act)
        torch.cuda.synchronize()
        yv = orc.decode(dt, y)
        assert np.isnan(yv[0])                                   # NaN in -> NaN out
        assert yv[5] == 0 and yv[6] == 0
        assert np.isfinite(yv[3:]).all() or dt == "f16"         # f16 may overflow for huge a*b
        dav, dbv = orc.decode(dt, to_bits(da, dt)), orc.decode(dt, to_bits(db, dt))
        assert np.isnan(dav[0]) and np.isnan(dbv[0])
        assert np.isfinite(dav[3:]).all() and np.isfinite(dbv[3:5]).all()
