"""Seeded random shapes of the gate/up GEMM with the activation in its
epilogue: single blocks and block pairs, every column-tile width, ragged row
and column tiles, K from one partial K step to several, strided and offset y;
every output against the oracle on operands whose sums are exact in fp32
(within 1 ulp)."""
import numpy as np
import pytest
import torch

import glu_activation_mlps_gb300 as glu
import glu_synth
from helpers import compare
from test_gemm_gpu import ACTS, DTYPES, cluster_size, expected_tiles, run_gemm

pytestmark = pytest.mark.gpu

N_CASES = 24


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    glu.build()
    glu.lib()


def random_case(i):
    rng = np.random.default_rng([2025, i])
    kind = i % 3
    if kind == 0:       # decode-sized rows: single blocks
        M, K, I = int(rng.integers(1, 129)), int(rng.integers(1, 49)) * 8, int(rng.integers(1, 3000))
    elif kind == 1:     # block pairs, a few tiles
        M, K, I = int(rng.integers(129, 1600)), int(rng.integers(1, 49)) * 8, int(rng.integers(1, 3000))
    else:               # many column tiles (the wider tile widths), short K
        M, K, I = int(rng.integers(1, 700)), int(rng.integers(1, 5)) * 8, int(rng.integers(8000, 40000))
    # keep the oracle's work (every output, two dot products of length K) small
    while M * I * K > 6e7:
        I = max(1, I // 2)
    y_pad = int(rng.integers(0, 3)) * 8 if rng.random() < 0.4 else 0
    return M, K, I, ACTS[i % 4], DTYPES[(i // 4) % 2], y_pad


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape(orc, i):
    M, K, I, act, dt, y_pad = random_case(i)
    rng = np.random.default_rng([31, i])
    x = glu_synth.grid_bits(rng, (M, K), dt)
    wg = glu_synth.grid_bits(rng, (I, K), dt)
    wu = glu_synth.grid_bits(rng, (I, K), dt)
    y, _, _ = run_gemm(x, wg, wu, dt, act, K, y_stride=I + y_pad if y_pad else None)
    info = glu.glu_last_launch()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert info["unroll"] == cluster_size(M, I) and info["vector_units"] == expected_tiles(M, I, sms)
    compare(y, orc.gemm_glu(act, dt, x, wg, wu), dt, what=f"case {i}: {M}x{K}x{I} {act} {dt} pad {y_pad}")
    assert glu.glu_wait_timeouts() == 0
