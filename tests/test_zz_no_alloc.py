"""glu_fwd_host_noalloc, the forward over host memory for callers that cannot
allocate device memory (a plug-in whose host application owns all device
memory, or a process that must not allocate once running): it stages rows in
a fixed array inside the library instead of a caller workspace.  Checked
through the C ABI against glu_fwd_host, the entry point it is a variant of,
on two calls in a row (the second must not see the first's leftovers); against
the oracle element by element in both layouts, every dtype, strided host rows
and in place over the up half; and for its size limit.  This file is
collected last."""
import numpy as np
import pytest
import torch

import glu_activation_mlps_gb300 as glu
import glu_synth
import oracle
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


# (layout, dtype, act, rows, cols, input row stride, output row stride or None for in place over
# the up half).  Strides are in elements; the f32 case has rows of 1.2 MB, so 27 rows fill the
# array and the 100 rows take four blocks.
WIDE_CASES = [
    ("split", "bf16", "gelu_tanh", 300, 2000, 2040, 2008),
    ("split", "f32", "silu", 100, 100000, 100000, 100000),
    ("split", "f16", "relu", 64, 4099, 4104, 4100),
    ("concat", "f16", "silu", 513, 3000, 6016, 3000),
    ("concat", "bf16", "gelu_erf", 200, 5000, 10008, None),
    ("concat", "f32", "gelu_tanh", 90, 1500, 3004, 1504),
]


def pinned(bits):
    signed = np.int32 if bits.dtype == np.uint32 else np.int16
    return torch.from_numpy(np.ascontiguousarray(bits).view(signed)).pin_memory()


@pytest.mark.parametrize("case", WIDE_CASES, ids=lambda c: f"{c[0]}-{c[1]}-{c[2]}-{c[3]}x{c[4]}")
def test_noalloc_against_the_oracle(case):
    """Both layouts, every dtype, host rows with padding between them (the
    row-by-row copies) and the [gate | up] forward written over the up half of
    its own host input: every element within the bar of the parity tests,
    the padding untouched, on two calls in a row with different inputs."""
    layout, dt, act, rows, cols, in_stride, out_stride = case
    s = torch.cuda.current_stream().cuda_stream
    bits_t = glu_synth.BITS_DTYPE[dt]
    sentinel = bits_t(0x7FAD) if dt != "f32" else bits_t(0x7FADBEEF)
    in_width = 2 * cols if layout == "concat" else cols
    for call in range(2):
        rng = np.random.default_rng([21, call, rows, cols])
        n_in = 1 if layout == "concat" else 2
        hosts, vals = [], []
        for _ in range(n_in):
            full = np.full((rows, in_stride), sentinel, dtype=bits_t)
            v = glu_synth.normal_bits(rng, (rows, in_width), 1.5, dt)
            full[:, :in_width] = v
            hosts.append(pinned(full))
            vals.append(v)
        if layout == "concat":
            want = oracle.fwd_concat(act, dt, vals[0], cols)
        else:
            want = oracle.fwd(act, dt, vals[0], vals[1])
        if out_stride is None:                       # in place over the up half of x
            y_host, y_ptr, ys = hosts[0], hosts[0].data_ptr() + cols * glu_synth.ELEM_BYTES[dt], in_stride
        else:
            y_host = pinned(np.full((rows, out_stride), sentinel, dtype=bits_t))
            y_ptr, ys = y_host.data_ptr(), out_stride
        b_ptr = hosts[1].data_ptr() if n_in == 2 else None
        st = glu.glu_fwd_host_noalloc(hosts[0].data_ptr(), in_stride, b_ptr, in_stride if n_in == 2 else 0,
                                      y_ptr, ys, rows, cols, glu.LAYOUT[layout], glu.ACT[act], glu.DTYPE[dt], s)
        assert st == 0, glu.glu_status_string(st) + " " + glu.glu_last_cuda_error()
        torch.cuda.current_stream().synchronize()
        out = y_host.numpy().view(bits_t)
        if out_stride is None:
            got = out[:, cols:2 * cols]
            assert np.array_equal(out[:, :cols], vals[0][:, :cols]), "the gate half changed"
            assert np.all(out[:, 2 * cols:] == sentinel), "padding written"
        else:
            got = out[:, :cols]
            assert np.all(out[:, cols:] == sentinel), "padding written"
        compare(got, want, dt, what=f"noalloc {layout} {dt} {act} call {call + 1}")
