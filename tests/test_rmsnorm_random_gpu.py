"""Seeded random configurations of the fused residual add + RMSNorm, forward
and backward, against the oracle: row counts that leave ragged stages and row
groups, widths on both sides of every kernel boundary (16-byte rows of 64 to
16384 elements, rows that are not 16-byte aligned), every dtype, with and
without dh and a second output, out of place and in place."""
import numpy as np
import pytest
import torch

import glu_activation_mlps_gb300 as glu
import glu_synth
from helpers import to_bits, to_dev
from test_rmsnorm_gpu import TORCH_INT_OF, bwd_inputs, check, check_bwd, inputs

pytestmark = pytest.mark.gpu

N_CASES = 48


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    glu.build()
    glu.lib()


def random_case(i):
    rng = np.random.default_rng([2024, i])
    dt = ("bf16", "f16", "f32")[i % 3]
    E = 4 if dt == "f32" else 2
    V = 16 // E
    kind = rng.integers(0, 4)
    if kind == 0:       # 16-byte rows up to 1024 vectors (the producer-warp kernel)
        H = int(rng.integers(1, 1024 // 2) * 2 * V) if rng.random() < 0.5 else int(rng.integers(1, 1025) * V)
    elif kind == 1:     # 16-byte rows past 1024 vectors
        H = int(rng.integers(1025, 2049) * V)
    elif kind == 2:     # rows that are not 16-byte aligned
        H = int(rng.integers(1, 4000)) | 1
    else:               # narrow rows
        H = int(rng.integers(1, 65) * V)
    rows = int(rng.integers(1, 3000 if H <= 4096 else 400))
    return dt, rows, H, bool(rng.random() < 0.5), bool(rng.random() < 0.3), bool(rng.random() < 0.3)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_forward_and_backward(orc, i):
    dt, rows, H, with_dh, dres, in_place = random_case(i)
    what = f"case {i}: {dt} {rows}x{H} dh={with_dh} dres={dres} in_place={in_place}"
    # forward
    x, r, g = inputs(rows, H, dt, 100 + i)
    xd, rd, gd = to_dev(x, dt), to_dev(r, dt), to_dev(g, dt)
    if in_place:
        h, y, rstd = glu.add_rmsnorm(xd, rd, gd, 1e-5, h=rd, y=xd, rstd=True)
    else:
        h, y, rstd = glu.add_rmsnorm(xd, rd, gd, 1e-5, rstd=True)
    torch.cuda.synchronize()
    check(orc, dt, x, r, g, 1e-5, to_bits(h, dt), to_bits(y, dt), rstd.cpu().numpy(), what + " forward")
    # backward
    dy, hb, rs, gb, dh = bwd_inputs(rows, H, dt, 200 + i, with_dh)
    dyd, hd, gbd = to_dev(dy, dt), to_dev(hb, dt), to_dev(gb, dt)
    dhd = to_dev(dh, dt) if with_dh else None
    rsd = torch.from_numpy(rs).cuda()
    dr = hd if (dres and in_place) else (torch.empty_like(dyd) if dres else None)
    dx_out = dyd if in_place else None
    dx, dgam = glu.add_rmsnorm_bwd(dyd, hd, rsd, gbd, dh=dhd, dx=dx_out, dres=dr, dgamma=True)
    torch.cuda.synchronize()
    if dr is not None:
        assert torch.equal(dr.view(TORCH_INT_OF[dt]), dx.view(TORCH_INT_OF[dt])), what + ": dres differs from dx"
    check_bwd(orc, dt, dy, hb, rs, gb, dh, to_bits(dx, dt), dgam.cpu().numpy(), what + " backward")
    assert glu.glu_wait_timeouts() == 0
