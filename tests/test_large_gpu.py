"""Maximum sizes: matrices with more than 2^32 elements (8.6 GB per bf16
operand), so that byte offsets need 64 bits and, on the element-wise path,
the unit -> row mapping takes its 64-bit branch.  Inputs are drawn on the
device from a seeded generator; the oracle checks a seeded sample of
elements plus the whole last row and the first elements."""
import numpy as np
import pytest
import torch

import glu_activation_mlps_gb300 as glu
from helpers import compare

pytestmark = pytest.mark.gpu

R = C = 65537                                  # 4 295 098 369 elements > 2^32


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    free, _ = torch.cuda.mem_get_info()
    if free < 60e9:
        pytest.skip("needs ~60 GB of free device memory")
    glu.build()
    glu.lib()
    yield
    glu.glu_set_tuning(0, 0, 0, 0, 0)
    torch.cuda.empty_cache()


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def sample_index(n_rows, n_cols):
    rng = np.random.default_rng(17)
    r = rng.integers(0, n_rows, 1 << 16)
    c = rng.integers(0, n_cols, 1 << 16)
    r = np.concatenate([r, np.full(n_cols, n_rows - 1), np.zeros(64, np.int64)])
    c = np.concatenate([c, np.arange(n_cols), np.arange(64)])
    return r, c


def gather(t2d, r, c):
    """Elements (r[i], c[i]) of a row-major matrix with any row stride."""
    n = (t2d.shape[0] - 1) * t2d.stride(0) + t2d.shape[1]
    flat = t2d.as_strided((n,), (1,))
    idx = torch.from_numpy(r * t2d.stride(0) + c).cuda()
    return bits(flat[idx])


@pytest.mark.parametrize("case", ["vector", "element"])
def test_forward_beyond_2_32_elements(orc, case):
    """vector: 65544 x 65544 with 16-byte aligned rows and a padded y stride,
    so 8193 units per row, 537 M units, byte offsets past 2^32.  element:
    65537 x 65537 (odd rows, no aligned access) on the element-wise path,
    whose 4.3 G elements take the 64-bit index branch."""
    n = 65544 if case == "vector" else R
    pad = 8 if case == "vector" else 1
    glu.glu_set_tuning(0 if case == "vector" else 2, 0, 0, 0, 0)
    g = torch.Generator(device="cuda").manual_seed(123)
    A = torch.empty(n, n, dtype=torch.bfloat16, device="cuda")
    B = torch.empty_like(A)
    for t in (A, B):                             # fill row blocks to bound the temporary
        for r0 in range(0, n, 8192):
            t[r0:r0 + 8192] = torch.randn(min(8192, n - r0), n, device="cuda", generator=g).to(torch.bfloat16)
    # y with a padded row stride: the rows are not contiguous in every operand
    Ybuf = torch.empty(n, n + pad, dtype=torch.bfloat16, device="cuda")
    Y = Ybuf[:, :n]
    glu.fwd(A, B, y=Y, act="silu")
    info = glu.glu_last_launch()
    assert info["flattened"] == 0
    if case == "vector":
        assert info["vec_bytes"] == 16 and info["vector_units"] == n * (n * 2 // 16)
    else:
        assert info["vector_units"] == 0 and info["tail_elems"] == n * n > 2 ** 32
    torch.cuda.synchronize()
    r, c = sample_index(n, n)
    a_s, b_s = gather(A, r, c), gather(B, r, c)
    compare(gather(Y, r, c), orc.fwd("silu", "bf16", a_s, b_s), "bf16", what=f"large fwd {case}")
    del A, B, Ybuf, Y
    torch.cuda.empty_cache()


def test_backward_beyond_2_32_elements_in_place(orc):
    glu.glu_set_tuning(0, 0, 0, 0, 0)
    g = torch.Generator(device="cuda").manual_seed(321)
    A, B, DC = (torch.empty(R, C, dtype=torch.bfloat16, device="cuda") for _ in range(3))
    for t in (A, B, DC):
        for r0 in range(0, R, 8192):
            t[r0:r0 + 8192] = torch.randn(min(8192, R - r0), C, device="cuda", generator=g).to(torch.bfloat16)
    r, c = sample_index(R, C)
    a_s, b_s, dc_s = gather(A, r, c), gather(B, r, c), gather(DC, r, c)
    glu.bwd(DC, A, B, inplace=True, act="gelu_tanh")
    info = glu.glu_last_launch()
    assert info["flattened"] == 1 and info["vector_units"] > 2 ** 28
    torch.cuda.synchronize()
    da_o, db_o = orc.bwd("gelu_tanh", "bf16", dc_s, a_s, b_s)
    compare(gather(A, r, c), da_o, "bf16", what="large bwd da")
    compare(gather(B, r, c), db_o, "bf16", what="large bwd db")
    del A, B, DC
    torch.cuda.empty_cache()
