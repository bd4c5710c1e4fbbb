"""The bounded wait that every staged kernel's mbarrier waits go through,
made to run out on the GPU: a warp waits on a barrier that nothing arrives
on.  The launch must return by itself after about a second, count one
timeout, and leave the context usable."""
import time

import numpy as np
import pytest
import torch

import glu_activation_mlps_gb300 as glu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    glu.build()
    glu.lib()


def test_wait_runs_out_and_context_stays_usable():
    torch.cuda.synchronize()
    glu.glu_wait_timeouts(reset=True)
    t0 = time.monotonic()
    glu.glu_wait_selftest()
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert glu.glu_wait_timeouts(reset=True) == 1
    assert 0.2 < elapsed < 10.0, f"the wait lasted {elapsed:.2f} s"
    # the context still runs kernels: a forward against torch
    a = torch.randn(64, 256, device="cuda")
    b = torch.randn(64, 256, device="cuda")
    y = glu.fwd(a, b, act="silu")
    torch.cuda.synchronize()
    ref = torch.nn.functional.silu(a.double()) * b.double()
    assert np.allclose(y.double().cpu().numpy(), ref.cpu().numpy(), rtol=1e-6, atol=1e-30)
    assert glu.glu_wait_timeouts() == 0
