"""The multi-GPU partition on one GPU: a batch split into contiguous blocks of
rows, one library call per block (what each rank of a data-parallel job does
with its shard, with no collective), must give exactly the bits of one call
over the whole batch, and those must meet the oracle's bar.

Shard bases fall at arbitrary byte offsets (odd widths, ragged shards), so the
shards take other access widths and row tails than the whole call: the
element results must not depend on where an element sits."""
import numpy as np
import pytest
import torch

import glu_activation_mlps_gb300 as glu
import glu_synth
import oracle
from helpers import compare, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    glu.build()
    glu.lib()
    glu.glu_set_tuning(0, 0, 0)


def shards(n_rows, parts):
    """Contiguous row blocks, sizes differing by at most one (the first ones larger)."""
    q, r = divmod(n_rows, parts)
    out, r0 = [], 0
    for k in range(parts):
        r1 = r0 + q + (1 if k < r else 0)
        out.append((r0, r1))
        r0 = r1
    return out


def test_shards_cover_the_rows_once():
    for n, g in ((1000, 7), (5, 8), (4096, 8), (3, 3)):
        sh = shards(n, g)
        assert sh[0][0] == 0 and sh[-1][1] == n
        assert all(a[1] == b[0] for a, b in zip(sh, sh[1:]))
        sizes = [b - a for a, b in sh]
        assert max(sizes) - min(sizes) <= 1


CASES = [
    ("silu", "bf16", "split", 1000, 4099, 7),
    ("gelu_erf", "f16", "split", 517, 2048, 3),
    ("gelu_tanh", "f32", "split", 300, 1025, 8),
    ("relu", "bf16", "concat", 640, 3001, 5),
    ("silu", "f16", "concat", 257, 11008, 2),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_row_shards_equal_the_whole_call(case):
    act, dt, layout, R, C, parts = case
    rng = np.random.default_rng([31, R, C, parts])
    width = 2 * C if layout == "concat" else C
    x = glu_synth.normal_bits(rng, (R, width), 2.0, dt)
    b = glu_synth.normal_bits(rng, (R, C), 1.0, dt)
    dc = glu_synth.normal_bits(rng, (R, C), 1.0, dt)
    X, B, DC = to_dev(x, dt), to_dev(b, dt), to_dev(dc, dt)
    split = layout == "split"
    # the whole batch
    y = glu.fwd(X, B if split else None, act=act, layout=layout)
    if split:
        da, db = glu.bwd(DC, X, B, act=act)
        dx = None
    else:
        dx = glu.bwd(DC, X, act=act, layout="concat")
    # one call per shard, into slices of preallocated outputs
    ys = torch.empty_like(y)
    das, dbs = (torch.empty_like(da), torch.empty_like(db)) if split else (None, None)
    dxs = None if split else torch.empty_like(dx)
    for r0, r1 in shards(R, parts):
        glu.fwd(X[r0:r1], B[r0:r1] if split else None, y=ys[r0:r1], act=act, layout=layout)
        if split:
            glu.bwd(DC[r0:r1], X[r0:r1], B[r0:r1], da=das[r0:r1], db=dbs[r0:r1], act=act)
        else:
            glu.bwd(DC[r0:r1], X[r0:r1], layout="concat", da=dxs[r0:r1], act=act)
    torch.cuda.synchronize()
    assert torch.equal(to_bits_t(y), to_bits_t(ys)), "forward shards differ from the whole call"
    if split:
        assert torch.equal(to_bits_t(da), to_bits_t(das)) and torch.equal(to_bits_t(db), to_bits_t(dbs))
    else:
        assert torch.equal(to_bits_t(dx), to_bits_t(dxs))
    # and the whole call against the oracle
    if split:
        compare(to_bits(ys, dt), oracle.fwd(act, dt, x, b), dt, what="shards y")
        da_o, db_o = oracle.bwd(act, dt, dc, x, b)
        scale = oracle.bwd_da_scale(act, dt, dc, x, b) if dt == "f32" else None
        compare(to_bits(das, dt), da_o, dt, scale=scale, what="shards da")
        compare(to_bits(dbs, dt), db_o, dt, what="shards db")
    else:
        compare(to_bits(ys, dt), oracle.fwd_concat(act, dt, x, C), dt, what="shards y")
        compare(to_bits(dxs, dt), oracle.bwd_concat(act, dt, dc, x, C), dt, what="shards dx")


def to_bits_t(t):
    return t.view(torch.int32 if t.dtype == torch.float32 else torch.int16)
