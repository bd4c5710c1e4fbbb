"""Guard bands: every output is placed inside a larger buffer filled with a
sentinel, and after the call every byte outside the output's elements (before,
after, and in the gaps between strided rows) must still hold the sentinel.
This is the check for the "unmasked tail corrupts adjacent memory" and
"off-by-one mask" failure modes of "Skill: Write a Triton SiLU-Mul (SwiGLU)
Kernel" (Correctness requirements; Common failure modes), run on odd widths,
misaligned bases and strides wider than the rows."""
import itertools

import numpy as np
import pytest
import torch

import glu_activation_mlps_gb300 as glu
import glu_synth
from helpers import compare, to_bits, to_dev

pytestmark = pytest.mark.gpu

TD = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
SENTINEL = {"f32": 0x7FBADBAD, "f16": 0x7DAD, "bf16": 0x7FAD}      # NaN patterns no kernel writes
INT = {"f32": torch.int32, "f16": torch.int16, "bf16": torch.int16}


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    glu.build()
    glu.lib()
    glu.glu_set_tuning(0, 0, 0)


def guarded(rows, cols, stride, offset, dt, guard=64):
    """(view, buffer, mask) where view is rows x cols at `offset` elements into
    a sentinel-filled buffer with row stride `stride`; mask marks the view's
    elements inside the buffer."""
    n = guard + offset + (rows - 1) * stride + cols + guard
    s = SENTINEL[dt]
    if dt != "f32" and s >= 0x8000:
        s -= 0x10000
    buf = torch.full((n,), s, dtype=INT[dt], device="cuda")
    start = guard + offset
    view = buf.view(TD[dt]).as_strided((rows, cols), (stride, 1), start)
    mask = np.zeros(n, dtype=bool)
    for r in range(rows):
        mask[start + r * stride: start + r * stride + cols] = True
    return view, buf, mask


def untouched(buf, mask, dt):
    bits = buf.cpu().numpy().view(np.uint32 if dt == "f32" else np.uint16)
    return bool((bits[~mask] == SENTINEL[dt]).all())


WIDTHS = (1, 7, 15, 16, 17, 1023, 11001)
CASES = list(itertools.product(WIDTHS, (1, 3), (0, 1, 3), (0, 1, 16)))


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_forward_writes_only_its_elements(orc, dt):
    for cols, rows, off, extra in CASES:
        rng = np.random.default_rng(cols * 31 + rows)
        a = glu_synth.normal_bits(rng, (rows, cols), 2.0, dt)
        b = glu_synth.normal_bits(rng, (rows, cols), 1.0, dt)
        A, B = to_dev(a, dt), to_dev(b, dt)
        Y, buf, mask = guarded(rows, cols, cols + extra, off, dt)
        glu.fwd(A, B, y=Y, act="gelu_tanh")
        assert untouched(buf, mask, dt), (cols, rows, off, extra)
        compare(to_bits(Y, dt), orc.fwd("gelu_tanh", dt, a, b), dt, what=f"{dt} {cols} {rows} {off} {extra}")


@pytest.mark.parametrize("dt", ["f16", "f32"])
def test_backward_writes_only_its_elements(orc, dt):
    for cols, rows, off, extra in CASES:
        rng = np.random.default_rng(cols * 17 + rows)
        a = glu_synth.normal_bits(rng, (rows, cols), 2.0, dt)
        b = glu_synth.normal_bits(rng, (rows, cols), 1.0, dt)
        dc = glu_synth.normal_bits(rng, (rows, cols), 1.0, dt)
        A, B, DC = to_dev(a, dt), to_dev(b, dt), to_dev(dc, dt)
        DA, bufa, ma = guarded(rows, cols, cols + extra, off, dt)
        DB, bufb, mb = guarded(rows, cols, cols + 2 * extra, (off + 1) % 4, dt)
        glu.bwd(DC, A, B, da=DA, db=DB, act="silu")
        assert untouched(bufa, ma, dt) and untouched(bufb, mb, dt), (cols, rows, off, extra)
        da_o, db_o = orc.bwd("silu", dt, dc, a, b)
        scale = orc.bwd_da_scale("silu", dt, dc, a, b) if dt == "f32" else None
        compare(to_bits(DA, dt), da_o, dt, scale=scale, what="da")
        compare(to_bits(DB, dt), db_o, dt, what="db")


def test_concat_inplace_leaves_the_gate_half_and_padding(orc):
    dt = "bf16"
    for cols in (5, 16, 1001, 1024):
        rows = 4
        rng = np.random.default_rng(cols)
        x = glu_synth.normal_bits(rng, (rows, 2 * cols), 1.5, dt)
        X, buf, _ = guarded(rows, 2 * cols, 2 * cols + 8, 0, dt)
        X.copy_(to_dev(x, dt))
        keep = buf.clone()
        glu.fwd(X, layout="concat", y=X[:, cols:], act="silu")
        after = buf.cpu().numpy()
        before = keep.cpu().numpy()
        guard = 64
        changed = np.flatnonzero(after != before)
        for i in changed:                          # every change is inside an up half
            r, c = divmod(i - guard, 2 * cols + 8)
            assert 0 <= r < rows and cols <= c < 2 * cols, (cols, i)
        compare(to_bits(X[:, cols:], dt), orc.fwd_concat("silu", dt, x, cols), dt, what=f"concat {cols}")
