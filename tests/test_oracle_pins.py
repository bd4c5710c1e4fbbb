"""Pins for the double-precision oracle (CPU only).

Each test checks the oracle against something other than itself: values and
constants printed on the pages (tests/golden/page_facts.json), closed forms,
invariants of the functions, central finite differences, an independent
arbitrary-precision evaluation of the pages' literal formulas (mpmath), and
library routines (torch fp64 activations and autograd, numpy's float16/float32
conversions, torch's float32->bfloat16 conversion).  A dropped term, a wrong
sign, a transposed operand or a wrong rounding in the oracle fails at least one.

Pages: "Skill: Write a Triton SiLU-Mul (SwiGLU) Kernel" (SM) and
"Kernel Profile: SwiGLU (Tier 1 - Element-wise)" (LP).
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import glu_synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")
ACTS = ("silu", "gelu_erf", "gelu_tanh", "relu")


@pytest.fixture(scope="module")
def facts():
    with open(GOLDEN) as f:
        return json.load(f)


def rel(x, y, scale=None):
    x, y = np.asarray(x, np.float64), np.asarray(y, np.float64)
    s = np.abs(y) if scale is None else np.asarray(scale)
    return np.max(np.abs(x - y) / np.maximum(s, 1e-300))


# --------------------------------------------------------------------------- closed forms

def test_closed_forms(orc):
    for a in ACTS:
        assert orc.act(a, [0.0])[0] == 0.0, a
        if a != "relu":
            # silu'(0) = sigmoid(0) = 1/2; gelu'(0) = Phi(0) = 1/2 (both forms)
            assert orc.act_grad(a, [0.0])[0] == 0.5, a
    # logistic(1) = e/(1+e) = 0.73105857863000487925...
    assert orc.act("silu", [1.0])[0] == pytest.approx(0.7310585786300048793, rel=1e-15)
    # silu(-88) = -88 e^-88/(1+e^-88) and its derivative e^-88 (1 - 87 + ...)/(...):
    # decimal values of the exact expressions
    assert orc.act("silu", [-88.0])[0] == pytest.approx(-5.328049667953043578e-37, rel=1e-13)
    assert orc.act_grad("silu", [-88.0])[0] == pytest.approx(-5.267503648999031720e-37, rel=1e-13)
    # relu and its subgradient choice (0 at 0)
    assert list(orc.act("relu", [-2.0, 0.0, 3.5])) == [0.0, 0.0, 3.5]
    assert list(orc.act_grad("relu", [-2.0, 0.0, 3.5])) == [0.0, 0.0, 1.0]


def test_silu_tends_to_identity_and_zero(orc):
    # silu(x) -> x for large x: 88 is a fixed point after rounding to bf16 and f32
    assert orc.round_to("bf16", orc.act("silu", [88.0]))[0] == 88.0
    assert orc.round_to("f32", orc.act("silu", [88.0]))[0] == 88.0
    # silu(x) -> 0- without NaN/inf for very negative x, including where exp(-x) overflows
    xs = np.array([-50.0, -100.0, -700.0, -710.0, -745.0, -1e4, -1e30, -3.4e38])
    for a in ACTS:
        for f in (orc.act, orc.act_grad):
            v = f(a, xs)
            assert np.all(np.isfinite(v)), (a, v)
            assert np.all(np.abs(v) < 1e-20), (a, v)
    assert np.all(orc.act("silu", xs) <= 0.0)


# --------------------------------------------------------------------------- invariants

def test_derivative_roots_and_silu_minimum(orc):
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    sig = lambda x: 1 / (1 + mp.e ** (-x))
    # roots of the pages' literal derivative formulas, solved at 40 digits
    r_silu = float(mp.findroot(lambda x: sig(x) + x * sig(x) * (1 - sig(x)), -1.28))
    r_erf = float(mp.findroot(lambda x: mp.ncdf(x) + x * mp.npdf(x), -0.75))
    k, c = mp.mpf("0.044715"), mp.sqrt(2 / mp.pi)
    gt = lambda x: 0.5 * x * (1 + mp.tanh(c * (x + k * x ** 3)))
    r_tanh = float(mp.findroot(lambda x: mp.diff(gt, x), -0.75))
    for name, r in (("silu", r_silu), ("gelu_erf", r_erf), ("gelu_tanh", r_tanh)):
        g = orc.act_grad(name, [r - 1e-7, r, r + 1e-7])
        assert g[0] < 0 < g[2], name            # the function's minimum: act' rises through 0
        assert abs(g[1]) < 1e-14, name
    # at the root of silu', 1 + a(1 - sigmoid(a)) = 0, so silu(a*) = a* + 1 (the minimum)
    assert orc.act("silu", [r_silu])[0] == pytest.approx(r_silu + 1.0, abs=1e-15)
    xs = np.linspace(-20, 20, 40001)
    assert orc.act("silu", xs).min() >= r_silu + 1.0 - 1e-15
    g = orc.act_grad("silu", xs)
    assert g.min() > -0.1 and g.max() < 1.1


def test_output_odd_in_b(orc):
    rng = np.random.default_rng(11)
    for dt in ("bf16", "f16", "f32"):
        a = glu_synth.normal_bits(rng, (257,), 2.0, dt)
        b = glu_synth.normal_bits(rng, (257,), 1.0, dt)
        dc = glu_synth.normal_bits(rng, (257,), 1.0, dt)
        sign = np.uint32(0x80000000) if dt == "f32" else np.uint16(0x8000)
        nb = b ^ sign
        for a_name in ACTS:
            y, yn = orc.fwd(a_name, dt, a, b), orc.fwd(a_name, dt, a, nb)
            assert np.array_equal(y ^ sign, yn) or np.array_equal(orc.decode(dt, y), -orc.decode(dt, yn))
            da, db = orc.bwd(a_name, dt, dc, a, b)
            dan, dbn = orc.bwd(a_name, dt, dc, a, nb)
            assert np.array_equal(orc.decode(dt, da), -orc.decode(dt, dan))
            assert np.array_equal(db, dbn)         # db does not depend on b


def test_activation_on_a_not_b(orc):
    """SM Correctness: the activation is applied to a (gate), not b (up)."""
    a = glu_synth.f32_to_bits(np.array([-1.0, 2.0, 0.5], np.float32), "f32")
    b = glu_synth.f32_to_bits(np.array([3.0, -0.25, 4.0], np.float32), "f32")
    y = orc.decode("f32", orc.fwd("silu", "f32", a, b))
    expect = np.array([3.0, -0.25, 4.0]) * np.array([-1.0, 2.0, 0.5]) / (1 + np.exp(-np.array([-1.0, 2.0, 0.5])))
    assert rel(y, expect) < 1e-7
    swapped = orc.decode("f32", orc.fwd("silu", "f32", b, a))
    assert rel(swapped, expect) > 1e-2


# --------------------------------------------------------------------------- page facts

def test_page_constants(facts):
    assert facts["erf_form_constant"]["value"] == pytest.approx(1 / math.sqrt(2), rel=1e-16)
    assert facts["tanh_form_cubic"]["value"] == 0.044715


def test_erf_and_tanh_forms_differ_as_stated(orc, facts):
    xs = np.linspace(-6, 6, 120001)
    d = np.abs(orc.act("gelu_erf", xs) - orc.act("gelu_tanh", xs))
    stated = facts["erf_vs_tanh_max_abs_diff"]["value"]
    assert 0.8 * stated < d.max() < 1.2 * stated      # "up to ~5e-4"
    assert d.max() > 1e-4                             # the two forms must differ


def test_silu_vs_gelu_gap(orc):
    """The printed 0.05 for max |silu - gelu_erf| on [-2, 2] is not what the
    functions give; the oracle must give the true 0.193 at x near -1.97."""
    xs = np.linspace(-2, 2, 400001)
    d = np.abs(orc.act("silu", xs) - orc.act("gelu_erf", xs))
    assert d.max() == pytest.approx(0.19335, abs=5e-4)
    assert xs[np.argmax(d)] == pytest.approx(-1.97, abs=0.05)


def test_three_printed_silu_derivative_forms(orc):
    """SM step 9: silu + sigmoid*(1 - silu); SM Correctness: sigmoid*(1 + a*(1 - sigmoid));
    LP gradient_formulas: silu*(1 - sigmoid) + sigmoid.  All three must equal the oracle."""
    from scipy.special import expit
    x = np.linspace(-30, 30, 60001)
    s = expit(x)
    silu = x * s
    forms = [silu + s * (1 - silu), s * (1 + x * (1 - s)), silu * (1 - s) + s]
    g = orc.act_grad("silu", x)
    t1, t2 = orc.act_grad_terms("silu", x)
    scale = np.abs(t1) + np.abs(t2) + 1e-300
    for f in forms:
        assert np.max(np.abs(f - g) / scale) < 1e-14


# --------------------------------------------------------------------------- finite differences

@pytest.mark.parametrize("name", ACTS)
def test_gradient_matches_central_differences(orc, name):
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.normal(0, 3, 3 * 7), np.linspace(-8, 8, 161)])
    if name == "relu":
        x = x[np.abs(x) > 1e-3]
    h = 1e-6 * np.maximum(1.0, np.abs(x))
    fd = (orc.act(name, x + h) - orc.act(name, x - h)) / (2 * h)
    g = orc.act_grad(name, x)
    t1, t2 = orc.act_grad_terms(name, x)
    assert np.max(np.abs(fd - g) / (np.abs(t1) + np.abs(t2) + 1e-12)) < 1e-7


def test_backward_elementwise_matches_finite_differences_of_forward(orc):
    """da = dc * d/da[act(a)*b], db = dc * d/db[act(a)*b] on a tiny 3x7 f32 case,
    checked with central differences of the forward formula in double."""
    rng = np.random.default_rng(5)
    for name in ACTS:
        a = glu_synth.normal_bits(rng, (3, 7), 2.0, "f32")
        b = glu_synth.normal_bits(rng, (3, 7), 1.0, "f32")
        dc = glu_synth.normal_bits(rng, (3, 7), 1.0, "f32")
        av, bv, cv = (orc.decode("f32", t) for t in (a, b, dc))
        if name == "relu":
            av = np.where(np.abs(av) < 1e-3, 0.5, av)
            a = orc.encode("f32", av)
        h = 1e-6
        f = lambda aa, bb: orc.act(name, aa) * bb
        fd_a = cv * (f(av + h, bv) - f(av - h, bv)) / (2 * h)
        fd_b = cv * (f(av, bv + h) - f(av, bv - h)) / (2 * h)
        da, db = orc.bwd(name, "f32", dc, a, b)
        m = orc.bwd_da_scale(name, "f32", dc, a, b)
        assert np.max(np.abs(orc.decode("f32", da) - fd_a) / (m + 1e-12)) < 1e-6
        assert np.max(np.abs(orc.decode("f32", db) - fd_b) / (np.abs(fd_b) + 1e-12)) < 1e-6


# --------------------------------------------------------------------------- arbitrary precision

def test_against_literal_page_formulas_at_high_precision(orc):
    """The oracle evaluates GeGLU-erf through erfc and GeGLU-tanh through a
    sigmoid; here the pages' literal erf/tanh formulas are evaluated at 130
    digits, enough to absorb their cancellation (1 + tanh(u) is ~1e-77 at the
    deepest point), down into the deep negative tails."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 130
    k, c = mp.mpf("0.044715"), mp.sqrt(2 / mp.pi)
    lit = {
        "silu": lambda x: x / (1 + mp.exp(-x)),
        "gelu_erf": lambda x: 0.5 * x * (1 + mp.erf(x / mp.sqrt(2))),
        "gelu_tanh": lambda x: 0.5 * x * (1 + mp.tanh(c * (x + k * x ** 3))),
    }
    lo = {"silu": -100.0, "gelu_erf": -14.0, "gelu_tanh": -13.0}
    for name, fn in lit.items():
        xs = np.concatenate([np.linspace(lo[name], 12, 397), [-1.27846, -0.7518, 1e-8, -1e-8]])
        want = np.array([float(fn(mp.mpf(float(x)))) for x in xs])
        got = orc.act(name, xs)
        assert rel(got, want) < 1e-12, name
        dwant = np.array([float(mp.diff(fn, mp.mpf(float(x)))) for x in xs[::4]])
        t1, t2 = orc.act_grad_terms(name, xs[::4])
        assert np.max(np.abs((t1 + t2) - dwant) / (np.abs(t1) + np.abs(t2))) < 1e-12, name


# the gate factor g of act(x) = x * g(x), as the pages print it, at high precision
def _gate_factors(mp):
    k, c = mp.mpf("0.044715"), mp.sqrt(2 / mp.pi)
    return {
        "silu": lambda x: 1 / (1 + mp.exp(-x)),                          # sigmoid
        "gelu_erf": lambda x: (1 + mp.erf(x / mp.sqrt(2))) / 2,          # Phi
        "gelu_tanh": lambda x: (1 + mp.tanh(c * (x + k * x ** 3))) / 2,
    }


def _split_points(name):
    roots = {"silu": -1.2784645427610738, "gelu_erf": -0.7517915246935645, "gelu_tanh": -0.7524614}
    lo = {"silu": -60.0, "gelu_erf": -12.0, "gelu_tanh": -11.0}[name]
    r = roots[name]
    return np.concatenate([np.linspace(lo, 12, 173), r + np.linspace(-1e-3, 1e-3, 11), [1e-9, -1e-9, 0.0]])


@pytest.mark.parametrize("name", ["silu", "gelu_erf", "gelu_tanh"])
def test_act_grad_terms_one_by_one(orc, name):
    """The oracle splits act'(x) of act(x) = x g(x) into t1 = g(x) and
    t2 = x g'(x) (product rule), and the fp32 tolerance of da scales with
    |t1| + |t2|.  Each term on its own, not only their sum, must equal the
    printed gate factor and x times its derivative, both evaluated here at
    60 digits with g' taken by mpmath's numerical differentiation of the
    printed g: sigmoid and x sigmoid(x) sigmoid(-x) for SiLU, Phi and x phi for
    GeGLU-erf, the tanh-form factor and x times its slope for GeGLU-tanh
    ("Kernel Profile: SwiGLU (Tier 1 - Element-wise)", Backward Pass,
    gradient formulas; "Skill: Write a Triton SiLU-Mul (SwiGLU) Kernel",
    Required reasoning process step 7).  A term moved from one side to the
    other, swapped or offset by a constant keeps the sum and fails here."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 60
    g = _gate_factors(mp)[name]
    xs = _split_points(name)
    want1 = np.array([float(g(mp.mpf(float(x)))) for x in xs])
    want2 = np.array([float(mp.mpf(float(x)) * mp.diff(g, mp.mpf(float(x)))) for x in xs])
    t1, t2 = orc.act_grad_terms(name, xs)
    assert np.max(np.abs(t1 - want1) / np.abs(want1)) < 1e-13, name
    nz = want2 != 0.0
    assert np.all(t2[~nz] == 0.0), name
    assert np.max(np.abs(t2[nz] - want2[nz]) / np.abs(want2[nz])) < 1e-12, name


def test_act_grad_terms_closed_values():
    """Closed forms of the split that need no numerical differentiation:
    SiLU at 0 is (1/2, 0); GeGLU-erf at 1 is (Phi(1), phi(1)) with
    Phi(1) = erfc(-1/sqrt 2)/2 and phi(1) = exp(-1/2)/sqrt(2 pi) (the
    standard normal CDF and density, here from scipy's ndtr and the textbook
    density); SiLU's t2 at x = ln 3 is ln 3 * (3/4) * (1/4); ReGLU's t2 is 0
    everywhere."""
    import oracle
    from scipy.special import ndtr
    t1, t2 = oracle.act_grad_terms("silu", [0.0, math.log(3.0)])
    assert (t1[0], t2[0]) == (0.5, 0.0)
    assert t1[1] == pytest.approx(0.75, rel=1e-15)
    assert t2[1] == pytest.approx(math.log(3.0) * 0.75 * 0.25, rel=1e-15)
    t1, t2 = oracle.act_grad_terms("gelu_erf", [1.0, -2.0])
    assert t1[0] == pytest.approx(ndtr(1.0), rel=1e-15)
    assert t2[0] == pytest.approx(math.exp(-0.5) / math.sqrt(2 * math.pi), rel=1e-15)
    assert t1[1] == pytest.approx(ndtr(-2.0), rel=1e-14)
    assert t2[1] == pytest.approx(-2.0 * math.exp(-2.0) / math.sqrt(2 * math.pi), rel=1e-15)
    x = np.array([-3.0, -0.0, 0.5, 7.0])
    t1, t2 = oracle.act_grad_terms("relu", x)
    assert list(t1) == [0.0, 0.0, 1.0, 1.0] and not np.any(t2)


@pytest.mark.parametrize("name", ACTS)
def test_bwd_da_scale_from_independent_terms(orc, name):
    """bwd_da_scale(dc, a, b) = |dc b| (|t1(a)| + |t2(a)|), rebuilt here from
    terms computed outside the oracle (mpmath as above; ReGLU: 1[a > 0], 0)
    on decoded bf16 inputs, every sign combination of dc and b included."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    rng = np.random.default_rng(11)
    n = 96
    a = glu_synth.normal_bits(rng, n, 2.0, "bf16")
    b = glu_synth.normal_bits(rng, n, 1.0, "bf16")
    dc = glu_synth.normal_bits(rng, n, 1.0, "bf16")
    av, bv, cv = (orc.decode("bf16", v) for v in (a, b, dc))
    if name == "relu":
        m1, m2 = (av > 0).astype(np.float64), np.zeros(n)
    else:
        g = _gate_factors(mp)[name]
        m1 = np.array([float(g(mp.mpf(float(x)))) for x in av])
        m2 = np.array([float(mp.mpf(float(x)) * mp.diff(g, mp.mpf(float(x)))) for x in av])
    want = np.abs(cv * bv) * (np.abs(m1) + np.abs(m2))
    got = orc.bwd_da_scale(name, "bf16", dc, a, b)
    assert np.all((got == 0) == (want == 0)), name
    nz = want != 0
    assert np.max(np.abs(got[nz] - want[nz]) / want[nz]) < 1e-12, name


# --------------------------------------------------------------------------- library routines

@pytest.mark.parametrize("name", ACTS)
def test_against_torch_fp64(orc, name):
    fn = {"silu": F.silu, "relu": F.relu,
          "gelu_erf": lambda t: F.gelu(t, approximate="none"),
          "gelu_tanh": lambda t: F.gelu(t, approximate="tanh")}[name]
    # torch's erf/tanh forms cancel for very negative x; stay where they are accurate
    lo = {"silu": -60.0, "relu": -60.0, "gelu_erf": -5.0, "gelu_tanh": -3.0}[name]
    x = np.concatenate([np.linspace(lo, 60, 24001), [0.0]])
    if name == "relu":
        x = x[x != 0.0]
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    y = fn(xt)
    (g,) = torch.autograd.grad(y.sum(), xt)
    t1, t2 = orc.act_grad_terms(name, x)
    scale = np.abs(t1) + np.abs(t2) + 1e-300
    yv = y.detach().numpy()
    # torch evaluates 0.5*x*(1 + erf|tanh(...)), whose rounding error is of order ulp(x)
    # where 1 + erf|tanh cancels; the oracle itself is pinned at 130 digits above
    yscale = np.abs(yv) + (np.abs(x) if name.startswith("gelu") else 0.0) + 1e-300
    assert rel(orc.act(name, x), yv, yscale) < 1e-12
    if name.startswith("gelu"):
        scale = scale + 1e-4      # torch's 0.5*(1 + erf|tanh) term carries ~1e-17 absolute error
    assert np.max(np.abs(orc.act_grad(name, x) - g.numpy()) / scale) < 1e-12


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_exhaustive_16bit_against_torch(orc, dt):
    """Every finite 16-bit a, b = dc = 1: rounded oracle outputs equal the
    rounded torch fp64 values wherever torch's own formula is accurate."""
    bits = glu_synth.all_finite_16bit(dt)
    a = orc.decode(dt, bits)
    one = orc.encode(dt, np.ones_like(a))
    for name, lo in (("silu", -700.0), ("relu", -np.inf), ("gelu_erf", -5.0), ("gelu_tanh", -3.0)):
        keep = a >= lo
        fn = {"silu": F.silu, "relu": F.relu,
              "gelu_erf": lambda t: F.gelu(t, approximate="none"),
              "gelu_tanh": lambda t: F.gelu(t, approximate="tanh")}[name]
        xt = torch.tensor(a[keep], dtype=torch.float64, requires_grad=True)
        y = fn(xt)
        (g,) = torch.autograd.grad(y.sum(), xt)
        val = lambda u: orc.decode(dt, u)           # compare values: +0 == -0
        y_or = orc.fwd(name, dt, bits[keep], one[keep])
        assert np.array_equal(val(y_or), orc.round_to(dt, y.detach().numpy())), name
        da, db = orc.bwd(name, dt, one[keep], bits[keep], one[keep])
        assert np.array_equal(db, y_or)
        g = g.numpy()
        if name == "relu":
            g = np.where(a[keep] == 0, 0.0, g)       # subgradient 0 at 0
        mism = val(da) != orc.round_to(dt, g)
        # rounding of a 1-ulp double difference can only flip a result that sits on a tie
        assert mism.sum() <= 2, (name, a[keep][mism])


def test_relu_product_is_the_exactly_rounded_product(orc):
    """ReGLU in bf16: relu(a)*b of two bf16 values is exact in float32, so
    torch's float32 product rounded once to bf16 must equal the oracle."""
    rng = np.random.default_rng(9)
    a = glu_synth.normal_bits(rng, (10000,), 3.0, "bf16")
    b = glu_synth.normal_bits(rng, (10000,), 3.0, "bf16")
    at = torch.from_numpy(a.astype(np.int16)).view(torch.bfloat16).float()
    bt = torch.from_numpy(b.astype(np.int16)).view(torch.bfloat16).float()
    want = (torch.relu(at) * bt).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = orc.fwd("relu", "bf16", a, b)
    nz = orc.decode("bf16", want) != 0                   # ignore the sign of zero
    assert np.array_equal(got[nz], want[nz])
    assert np.all(orc.decode("bf16", got[~nz]) == 0)


# --------------------------------------------------------------------------- rounding and codecs

def _random_doubles(rng, n, lo_exp, hi_exp):
    m = rng.uniform(1.0, 2.0, n)
    e = rng.integers(lo_exp, hi_exp, n)
    s = rng.choice([-1.0, 1.0], n)
    return s * np.ldexp(m, e)


def test_f16_rounding_matches_numpy(orc):
    rng = np.random.default_rng(1)
    x = _random_doubles(rng, 200000, -30, 18)
    # exact midpoints between neighbouring f16 values (ties) and the overflow edge
    h = np.arange(0, 0x7BFF, 7, dtype=np.uint16).view(np.float16).astype(np.float64)
    hn = (np.arange(0, 0x7BFF, 7, dtype=np.uint16) + 1).view(np.float16).astype(np.float64)
    x = np.concatenate([x, (h + hn) / 2, -(h + hn) / 2, [65504.0, 65519.99, 65520.0, 1e6, 2.0 ** -25, 2.0 ** -26]])
    want = x.astype(np.float16)
    assert np.array_equal(orc.encode("f16", x), want.view(np.uint16))
    assert np.array_equal(orc.round_to("f16", x), want.astype(np.float64))


def test_f32_rounding_matches_numpy(orc):
    rng = np.random.default_rng(2)
    x = _random_doubles(rng, 200000, -160, 130)
    f = np.arange(1, 1 << 20, 997, dtype=np.uint32).view(np.float32).astype(np.float64)
    fn = (np.arange(1, 1 << 20, 997, dtype=np.uint32) + 1).view(np.float32).astype(np.float64)
    with np.errstate(over="ignore"):
        x = np.concatenate([x, (f + fn) / 2, [3.5e38, 3.402823466385289e38]])
        want = x.astype(np.float32)
    assert np.array_equal(orc.encode("f32", x), want.view(np.uint32))


def test_bf16_rounding(orc):
    rng = np.random.default_rng(3)
    # (1) doubles that are float32 values: torch's float32 -> bfloat16 is one RNE
    f = rng.standard_normal(200000).astype(np.float32) * np.float32(1e3)
    f = np.concatenate([f, np.arange(0, 1 << 20, 3, dtype=np.uint32).view(np.float32)])  # tiny/subnormal
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    assert np.array_equal(orc.encode("bf16", f.astype(np.float64)), want)
    # (2) general doubles: the result is a bf16 value, no neighbour is nearer, ties go to even
    x = _random_doubles(rng, 100000, -140, 128)
    u = orc.encode("bf16", x)
    r = orc.decode("bf16", u)
    up = orc.decode("bf16", u + np.uint16(1))
    dn = orc.decode("bf16", np.where((u & 0x7FFF) > 0, u - np.uint16(1), u))
    fin = np.isfinite(up) & np.isfinite(dn) & np.isfinite(r)
    err = np.abs(x - r)
    assert np.all(err[fin] <= np.abs(x - up)[fin])
    assert np.all(err[fin] <= np.abs(x - dn)[fin])
    tie = fin & ((err == np.abs(x - up)) | (err == np.abs(x - dn))) & (err > 0)
    assert np.all((u[tie] & 1) == 0)


def test_decode_all_16bit_patterns(orc):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    h = bits.view(np.float16).astype(np.float64)
    d = orc.decode("f16", bits)
    ok = ~np.isnan(h)
    assert np.array_equal(d[ok], h[ok]) and np.all(np.isnan(d[~ok]))
    bt = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).double().numpy()
    d = orc.decode("bf16", bits)
    ok = ~np.isnan(bt)
    assert np.array_equal(d[ok], bt[ok]) and np.all(np.isnan(d[~ok]))
    for dt in ("f16", "bf16"):
        fin = glu_synth.all_finite_16bit(dt)
        assert np.array_equal(orc.encode(dt, orc.decode(dt, fin)), fin)


# --------------------------------------------------------------------------- layouts

def test_concat_layout_is_gate_then_up(orc):
    rng = np.random.default_rng(4)
    x = glu_synth.normal_bits(rng, (5, 2 * 9), 1.0, "bf16")
    y = orc.fwd_concat("silu", "bf16", x, 9)
    assert np.array_equal(y, orc.fwd("silu", "bf16", x[:, :9], x[:, 9:]))
    dc = glu_synth.normal_bits(rng, (5, 9), 1.0, "bf16")
    dx = orc.bwd_concat("silu", "bf16", dc, x, 9)
    da, db = orc.bwd("silu", "bf16", dc, x[:, :9], x[:, 9:])
    assert np.array_equal(dx[:, :9], da) and np.array_equal(dx[:, 9:], db)


def test_threaded_drivers_equal_serial(orc):
    d = glu_synth.sweep(1024, "bf16", rows=64)
    y1 = orc.fwd("gelu_erf", "bf16", d["a"], d["b"])
    y2 = orc.fwd_threaded("gelu_erf", "bf16", d["a"], d["b"], threads=4)
    assert np.array_equal(y1, y2)
    g1 = orc.bwd("gelu_tanh", "bf16", d["dc"], d["a"], d["b"])
    g2 = orc.bwd_threaded("gelu_tanh", "bf16", d["dc"], d["a"], d["b"], threads=3)
    assert all(np.array_equal(p, q) for p, q in zip(g1, g2))


# --------------------------------------------------------------------------- gate/up projections

def test_gemm_glu_gate_and_up_match_numpy_matmul(orc):
    """g and u are the projections x @ w^T: checked against numpy's float64
    matmul, and y against the element-wise oracle applied to them."""
    rng = np.random.default_rng(41)
    M, K, I = 7, 96, 11
    x = glu_synth.normal_bits(rng, (M, K), 1.0, "bf16")
    wg = glu_synth.normal_bits(rng, (I, K), 0.1, "bf16")
    wu = glu_synth.normal_bits(rng, (I, K), 0.1, "bf16")
    xv, gv, uv = (orc.decode("bf16", t) for t in (x, wg, wu))
    mm, ii = np.meshgrid(np.arange(M), np.arange(I), indexing="ij")
    y, g, u, sg, su = orc.gemm_glu_at("silu", "bf16", x, wg, wu, mm.ravel(), ii.ravel())
    assert np.allclose(g, (xv @ gv.T).ravel(), rtol=1e-13, atol=1e-13)
    assert np.allclose(u, (xv @ uv.T).ravel(), rtol=1e-13, atol=1e-13)
    assert np.allclose(sg, (np.abs(xv) @ np.abs(gv).T).ravel(), rtol=1e-13)
    want = orc.round_to("bf16", orc.act("silu", g) * u)
    assert np.array_equal(orc.decode("bf16", y), want)
    # row i of the weights is output feature i: swapping the operands changes the result
    y_sw, *_ = orc.gemm_glu_at("silu", "bf16", x, wu, wg, mm.ravel(), ii.ravel())
    assert not np.array_equal(y, y_sw)


def test_gemm_glu_exact_integer_case(orc):
    """Small integers: every product and sum is exact, so g and u are known in
    closed form (x = 1, weights = k-index pattern)."""
    K = 8
    x = orc.encode("bf16", np.ones((1, K)))
    wg = orc.encode("bf16", np.arange(K, dtype=float)[None, :] - 3.0)       # sum = 28 - 24 = 4
    wu = orc.encode("bf16", np.full((1, K), 0.5))                            # sum = 4
    y, g, u, *_ = orc.gemm_glu_at("relu", "bf16", x, wg, wu, [0], [0])
    assert g[0] == 4.0 and u[0] == 4.0 and orc.decode("bf16", y)[0] == 16.0
    y2 = orc.gemm_glu("gelu_tanh", "bf16", x, wg, wu)
    assert orc.decode("bf16", y2)[0, 0] == orc.round_to("bf16", orc.act("gelu_tanh", [4.0]) * 4.0)[0]


# --------------------------------------------------------------------------- the MLP's down projection
# "Fused Kernels", section 4, "The fused MLP"; the product y @ w_down^T.

def test_matmul_nt_matches_numpy(orc):
    """d = a b^T against numpy's float64 matmul of the decoded operands, both
    the exact sum and its one rounding, at scattered (m, n) pairs; operand
    order matters (b a^T differs)."""
    rng = np.random.default_rng(41)
    M, N, K = 9, 13, 300
    for dt in ("bf16", "f16"):
        a = glu_synth.normal_bits(rng, (M, K), 1.0, dt)
        b = glu_synth.normal_bits(rng, (N, K), 1.0, dt)
        A, B = orc.decode(dt, a), orc.decode(dt, b)
        ref = A @ B.T
        ms, ns = rng.integers(0, M, 40), rng.integers(0, N, 40)
        d, ex, sa = orc.matmul_nt_at(dt, a, b, ms, ns)
        want = ref[ms, ns]
        assert np.all(np.abs(ex - want) <= 1e-13 * (np.abs(A[ms]) @ np.abs(B).T)[np.arange(40), ns])
        assert np.allclose(sa, (np.abs(A[ms]) * np.abs(B[ns])).sum(1), rtol=1e-14, atol=0)
        assert np.array_equal(d, orc.encode(dt, ex))
        # the transposed order reads other rows: different values where the shapes allow
        d2, ex2, _ = orc.matmul_nt_at(dt, b[:M], a[:M], ms % M, ns % M)
        assert not np.allclose(ex2, ex)


def test_matmul_nt_integer_closed_form(orc):
    """a[m, k] = m + 1, b[n, k] = k - n: d[m, n] = (m + 1) (K (K - 1) / 2 - n K), exact."""
    M, N, K = 3, 4, 16
    a = orc.encode("bf16", np.repeat(np.arange(1, M + 1, dtype=float)[:, None], K, 1))
    b = orc.encode("bf16", np.arange(K, dtype=float)[None, :] - np.arange(N, dtype=float)[:, None])
    mm, nn = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    d, ex, _ = orc.matmul_nt_at("bf16", a, b, mm.ravel(), nn.ravel())
    want = (mm.ravel() + 1) * (K * (K - 1) / 2 - nn.ravel() * K)
    assert np.array_equal(ex, want) and np.array_equal(orc.decode("bf16", d), want)


def test_mlp_is_the_two_products(orc):
    """mlp() = the gated first half rounded to the dtype, then the down
    projection of that stored y (numpy's matmul of the decoded y)."""
    rng = np.random.default_rng(42)
    M, Hd, I = 6, 40, 24
    x = glu_synth.normal_bits(rng, (M, Hd), 1.0, "bf16")
    wg, wu = (glu_synth.normal_bits(rng, (I, Hd), 0.2, "bf16") for _ in range(2))
    wd = glu_synth.normal_bits(rng, (Hd, I), 0.2, "bf16")
    out, y, ex, sa = orc.mlp("silu", "bf16", x, wg, wu, wd)
    assert np.array_equal(y, orc.gemm_glu("silu", "bf16", x, wg, wu))
    ref = orc.decode("bf16", y) @ orc.decode("bf16", wd).T
    assert np.allclose(ex, ref, rtol=0, atol=1e-13 * sa.max())
    assert np.array_equal(out, orc.encode("bf16", ex))


# --------------------------------------------------------------------------- residual add + RMSNorm
# Page: "Skill: Write a Triton Fused Add+RMSNorm Kernel" (AR).

def _bf16(v):
    return glu_synth.f32_to_bits(np.asarray(v, dtype=np.float32), "bf16")


def test_add_rmsnorm_constant_row_closed_form(orc):
    """A constant row h = c: mean square c^2, so rstd = 1/sqrt(c^2 + eps) and
    y = c * rstd * gamma.  With eps = 1 the eps-inside-the-root form of (AR)
    Kernel design rules (1.75/sqrt(1.75^2 + 1) = 0.868) differs from eps outside
    (1.75/2.75) and from a mean-subtracting norm (0)."""
    H = 6
    x = _bf16(np.full((1, H), 1.5))
    r = _bf16(np.full((1, H), 0.25))
    g = _bf16(np.full(H, 2.0))
    h, y, rstd, ye = orc.add_rmsnorm("bf16", x, r, g, 1.0)
    want = 1.0 / math.sqrt(1.75 ** 2 + 1.0)
    assert rstd[0] == pytest.approx(want, rel=1e-15)
    assert np.allclose(ye, 1.75 * want * 2.0, rtol=1e-15, atol=0)
    assert np.all(orc.decode("bf16", h) == 1.75)


def test_add_rmsnorm_unit_rms_identity(orc):
    """rstd^2 * mean(h^2) + eps * rstd^2 = 1, i.e. mean((y/gamma)^2) + eps*rstd^2 = 1
    for every row: fixes the denominator H and the placement of eps."""
    rng = np.random.default_rng(50)
    rows, H = 5, 777
    x = glu_synth.normal_bits(rng, (rows, H), 1.0, "bf16")
    r = glu_synth.normal_bits(rng, (rows, H), 3.0, "bf16")
    g = glu_synth.normal_bits(rng, H, 1.0, "bf16")
    gv = orc.decode("bf16", g)
    for eps in (1e-6, 0.5, 7.0):
        _, _, rstd, ye = orc.add_rmsnorm("bf16", x, r, g, eps)
        lhs = np.mean((ye / gv) ** 2, axis=1) + eps * rstd ** 2
        assert np.allclose(lhs, 1.0, rtol=0, atol=1e-13)


def test_add_rmsnorm_gamma_is_per_column(orc):
    """y[r, j] / (h[r, j] * gamma[j]) is the same rstd[r] for every column j of
    every row ((AR) step 6: gamma indexed by the column only)."""
    rng = np.random.default_rng(51)
    rows, H = 4, 64
    x = glu_synth.normal_bits(rng, (rows, H), 1.0, "f16")
    r = glu_synth.normal_bits(rng, (rows, H), 1.0, "f16")
    g = glu_synth.f32_to_bits(np.linspace(0.5, 3.0, H, dtype=np.float32), "f16")
    _, _, rstd, ye = orc.add_rmsnorm("f16", x, r, g, 1e-5)
    h = orc.decode("f16", x) + orc.decode("f16", r)
    ratio = ye / (h * orc.decode("f16", g)[None, :])
    assert np.allclose(ratio, rstd[:, None], rtol=1e-14, atol=0)
    assert len(set(np.round(rstd, 12))) == rows


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
def test_add_rmsnorm_stored_sum_is_the_rounded_sum(orc, dt):
    """The stored h is x + res rounded once ((AR) step 4): checked against
    numpy's float16/float32 and torch's bfloat16 conversion of the float64 sum."""
    rng = np.random.default_rng(52)
    x = glu_synth.normal_bits(rng, (3, 500), 1.0, dt)
    r = glu_synth.normal_bits(rng, (3, 500), 50.0, dt)
    g = glu_synth.normal_bits(rng, 500, 1.0, dt)
    h, *_ = orc.add_rmsnorm(dt, x, r, g, 1e-6)
    s = orc.decode(dt, x) + orc.decode(dt, r)
    if dt == "f16":
        want = s.astype(np.float16).view(np.uint16)
    elif dt == "f32":
        want = s.astype(np.float32).view(np.uint32)
    else:
        want = torch.from_numpy(s).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(h, want)


def test_add_rmsnorm_squares_the_exact_sum(orc):
    """(AR) step 3: the add runs before any narrowing.  x = (1, 1), res = (2^-9, 0)
    in bf16: the exact h = (1 + 2^-9, 1) is not a bf16 pair (the stored h is
    (1, 1)), and the mean square is that of the exact h."""
    x = _bf16([[1.0, 1.0]])
    r = _bf16([[2.0 ** -9, 0.0]])
    g = _bf16([1.0, 1.0])
    eps = 1e-6
    h, _, rstd, ye = orc.add_rmsnorm("bf16", x, r, g, eps)
    assert np.all(orc.decode("bf16", h) == 1.0)
    ms = ((1 + 2.0 ** -9) ** 2 + 1.0) / 2
    assert rstd[0] == pytest.approx(1 / math.sqrt(ms + eps), rel=1e-15)
    assert ye[0, 1] == pytest.approx(1 / math.sqrt(ms + eps), rel=1e-15)
    assert ye[0, 1] != pytest.approx(1 / math.sqrt(1.0 + eps), rel=1e-8)


def test_add_rmsnorm_matches_torch_rms_norm(orc):
    """torch.nn.functional.rms_norm in float64 on x + res with weight gamma."""
    if not hasattr(F, "rms_norm"):
        pytest.skip("torch without rms_norm")
    rng = np.random.default_rng(53)
    rows, H = 6, 4096
    x = glu_synth.normal_bits(rng, (rows, H), 1.0, "bf16")
    r = glu_synth.normal_bits(rng, (rows, H), 2.0, "bf16")
    g = glu_synth.normal_bits(rng, H, 0.3, "bf16")
    _, y, _, ye = orc.add_rmsnorm("bf16", x, r, g, 1e-5)
    h = torch.from_numpy(orc.decode("bf16", x) + orc.decode("bf16", r))
    want = F.rms_norm(h, (H,), weight=torch.from_numpy(orc.decode("bf16", g)), eps=1e-5).numpy()
    assert np.allclose(ye, want, rtol=1e-12, atol=1e-300)
    assert np.array_equal(orc.decode("bf16", y), orc.round_to("bf16", want))


def test_add_rmsnorm_scale_invariance(orc):
    """Scaling x and res by 2^k and eps by 4^k leaves y unchanged (exact in bf16)."""
    rng = np.random.default_rng(54)
    x = glu_synth.normal_bits(rng, (3, 300), 1.0, "bf16")
    r = glu_synth.normal_bits(rng, (3, 300), 1.0, "bf16")
    g = glu_synth.normal_bits(rng, 300, 1.0, "bf16")
    _, _, _, ye = orc.add_rmsnorm("bf16", x, r, g, 1e-3)
    xs = _bf16(orc.decode("bf16", x) * 2.0 ** 40)
    rs = _bf16(orc.decode("bf16", r) * 2.0 ** 40)
    _, _, _, ye2 = orc.add_rmsnorm("bf16", xs, rs, g, 1e-3 * 2.0 ** 80)
    assert np.allclose(ye, ye2, rtol=1e-14, atol=0)


def _rmsnorm_setup(rng, rows, H, dt, eps):
    h = glu_synth.normal_bits(rng, (rows, H), 3.0, dt)
    dy = glu_synth.normal_bits(rng, (rows, H), 1.0, dt)
    g = glu_synth.f32_to_bits(rng.standard_normal(H, dtype=np.float32) * np.float32(0.2) + np.float32(1.0), dt)
    return h, dy, g


def _exact_rstd(orc, dt, h, g, eps):
    zero = np.zeros_like(h)
    _, _, rstd, _ = orc.add_rmsnorm(dt, h, zero, g, eps)
    return rstd


def test_add_rmsnorm_bwd_matches_torch_autograd(orc):
    """ds and dgamma against torch's float64 autograd through F.rms_norm, with
    the rstd the forward keeps (fp32) in place of torch's own."""
    if not hasattr(F, "rms_norm"):
        pytest.skip("torch without rms_norm")
    rng = np.random.default_rng(60)
    rows, H, eps = 4, 1024, 1e-5
    h, dy, g = _rmsnorm_setup(rng, rows, H, "bf16", eps)
    rstd = _exact_rstd(orc, "bf16", h, g, eps)
    _, ds, dgamma = orc.add_rmsnorm_bwd("bf16", dy, h, rstd.astype(np.float32), g)
    ht = torch.tensor(orc.decode("bf16", h), requires_grad=True)
    gt = torch.tensor(orc.decode("bf16", g), requires_grad=True)
    y = F.rms_norm(ht, (H,), weight=gt, eps=eps)
    y.backward(torch.tensor(orc.decode("bf16", dy)))
    scale = np.abs(ht.grad.numpy()).max()
    assert np.allclose(ds, ht.grad.numpy(), rtol=1e-6, atol=1e-6 * scale)
    assert np.allclose(dgamma, gt.grad.numpy(), rtol=1e-6, atol=1e-6 * np.abs(gt.grad.numpy()).max())


def test_add_rmsnorm_bwd_finite_differences(orc):
    """ds is the derivative of L = sum(dy * y) along h (central differences of
    the forward oracle in f32 with steps of 2^-12 |h|)."""
    rng = np.random.default_rng(61)
    H, eps = 48, 0.3
    h, dy, g = _rmsnorm_setup(rng, 1, H, "f32", eps)
    rstd = _exact_rstd(orc, "f32", h, g, eps)
    _, ds, _ = orc.add_rmsnorm_bwd("f32", dy, h, rstd.astype(np.float32), g)
    hv = orc.decode("f32", h)[0]
    dyv = orc.decode("f32", dy)[0]
    zero = np.zeros((1, H), dtype=np.uint32)
    for j in (0, 7, 31, 47):
        step = 2.0 ** (np.floor(np.log2(abs(hv[j]))) - 12)
        vals = []
        for sgn in (1, -1):
            hp = hv.copy()
            hp[j] += sgn * step
            _, _, _, ye = orc.add_rmsnorm("f32", glu_synth.f32_to_bits(hp[None, :].astype(np.float32), "f32"), zero,
                                          g, eps)
            vals.append(float(np.dot(dyv, ye[0])))
        fd = (vals[0] - vals[1]) / (2 * step)
        assert fd == pytest.approx(ds[0, j], rel=2e-5, abs=1e-6)


def test_add_rmsnorm_bwd_identities(orc):
    """sum_j ds_j s_j = rstd D (1 - rstd^2 mean(s^2)) with D = sum gamma dy s (the
    gradient along s only rescales the norm term); dh is added unchanged; dgamma
    sums its rows."""
    rng = np.random.default_rng(62)
    rows, H, eps = 3, 200, 1e-2
    h, dy, g = _rmsnorm_setup(rng, rows, H, "f16", eps)
    rstd = _exact_rstd(orc, "f16", h, g, eps).astype(np.float32)
    _, ds, dgamma = orc.add_rmsnorm_bwd("f16", dy, h, rstd, g)
    s, d, gv, rs = orc.decode("f16", h), orc.decode("f16", dy), orc.decode("f16", g), rstd.astype(np.float64)
    D = np.sum(gv[None, :] * d * s, axis=1)
    ms = np.mean(s * s, axis=1)
    assert np.allclose(np.sum(ds * s, axis=1), rs * D * (1 - rs * rs * ms), rtol=1e-9, atol=1e-12)
    dh = glu_synth.normal_bits(rng, (rows, H), 1.0, "f16")
    _, ds2, dgamma2 = orc.add_rmsnorm_bwd("f16", dy, h, rstd, g, dh)
    assert np.allclose(ds2 - ds, orc.decode("f16", dh), rtol=0, atol=1e-12)
    assert np.array_equal(dgamma, dgamma2)
    parts = [orc.add_rmsnorm_bwd("f16", dy[r:r + 1], h[r:r + 1], rstd[r:r + 1], g)[2] for r in range(rows)]
    assert np.allclose(dgamma, np.sum(parts, axis=0), rtol=1e-14, atol=0)
