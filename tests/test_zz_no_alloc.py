"""glu_fwd_host_noalloc, the forward over host memory for callers that cannot
allocate device memory (a plug-in whose host application owns all device
memory, or a process that must not allocate once running): it stages rows in
a fixed array inside the library instead of a caller workspace.  Checked
through the C ABI against glu_fwd_host, the entry point it is a variant of,
on two calls in a row (the second must not see the first's leftovers), and
for its size limit.  This file is collected last."""
import numpy as np
import pytest
import torch

import glu_activation_mlps_gb300 as glu
import glu_synth
from helpers import compare

pytestmark = pytest.mark.gpu

SCRATCH = 32 * 1024 * 1024


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    glu.build()
    glu.lib()


def host_bits(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).pin_memory()


def reference_fwd(a, b, rows, cols, act):
    """The same forward through glu_fwd_host with a caller workspace."""
    y = torch.empty((rows, cols), dtype=torch.int16).pin_memory()
    need = glu.glu_host_workspace_bytes(64, cols, 0, glu.DTYPE["bf16"], 0)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = glu.glu_fwd_host(a.data_ptr(), cols, b.data_ptr(), cols, y.data_ptr(), cols, rows, cols, 0,
                          glu.ACT[act], glu.DTYPE["bf16"], ws.data_ptr(), need, s, s, s)
    assert st == 0
    torch.cuda.current_stream().synchronize()
    return y.numpy().view(np.uint16)


def test_noalloc_matches_glu_fwd_host_on_two_calls():
    s = torch.cuda.current_stream().cuda_stream
    # a row of 3 x 14336 bf16 is 86 KiB, so 4096 rows need many blocks of the array
    for call, (rows, cols, act, seed) in enumerate(((4096, 14336, "silu", 11), (777, 4001, "gelu_erf", 12))):
        rng = np.random.default_rng(seed)
        a = host_bits(glu_synth.normal_bits(rng, (rows, cols), 2.0, "bf16"))
        b = host_bits(glu_synth.normal_bits(rng, (rows, cols), 1.0, "bf16"))
        y = torch.full((rows, cols), 0x7FAD, dtype=torch.int16).pin_memory()
        st = glu.glu_fwd_host_noalloc(a.data_ptr(), cols, b.data_ptr(), cols, y.data_ptr(), cols, rows, cols,
                                      0, glu.ACT[act], glu.DTYPE["bf16"], s)
        assert st == 0, glu.glu_status_string(st)
        torch.cuda.current_stream().synchronize()
        want = reference_fwd(a, b, rows, cols, act)
        stats = compare(y.numpy().view(np.uint16), want, "bf16", what=f"noalloc call {call + 1}")
        assert stats["max_ulp"] == 0          # the same kernels: identical bits


def test_noalloc_rejects_rows_that_do_not_fit():
    s = torch.cuda.current_stream().cuda_stream
    cols = SCRATCH // 6 + 1                   # one row of a, b and y: 3 * 2 bytes per column
    a, b, y = (torch.zeros((2, cols), dtype=torch.int16) for _ in range(3))
    st = glu.glu_fwd_host_noalloc(a.data_ptr(), cols, b.data_ptr(), cols, y.data_ptr(), cols, 2, cols, 0, 0,
                                  glu.DTYPE["bf16"], s)
    assert st == -7 and "workspace" in glu.glu_status_string(st)
    assert (y == 0).all()                     # nothing was written
