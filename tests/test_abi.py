"""The C-ABI library on the CPU: it loads, exports every symbol include/glu.h
declares, and its host-side validation returns the documented status codes.

No test here enqueues GPU work.  Fake device addresses are only ever passed to
calls that must be rejected before any launch, and every test that passes them
(including those that let a valid call reach the CUDA runtime, which fails for
want of a device) is skipped whenever a GPU is present."""
import os
import re
import subprocess

import pytest
import torch

import glu_activation_mlps_gb300 as glu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "glu.h")

OK, NULL, SHAPE, STRIDE, ALIAS, ENUM, CUDA, WORKSPACE = 0, -1, -2, -3, -4, -5, -6, -7
SPLIT, CONCAT = 0, 1
SILU, RELU = 0, 3
F32, F16, BF16 = 0, 1, 2
BASE = 1 << 32          # fake, 4 KiB-aligned device addresses: never dereferenced

# Tests that pass fake device addresses run only where no GPU is present: on a
# GPU a validation mistake would launch a kernel on them.
cpu_only = pytest.mark.skipif(torch.cuda.is_available(), reason="passes fake device addresses")


@pytest.fixture(scope="module", autouse=True)
def built():
    glu.build()
    glu.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(glu_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol():
    names = declared_functions()
    assert set(names) == set(glu.EXPORTS)
    out = subprocess.run(["nm", "-D", "--defined-only", glu.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (glu_\w+)", out))
    for n in names:
        assert n in exported, n
        assert hasattr(glu.lib(), n)


def test_version_matches_header():
    v = int(re.search(r"#define GLU_VERSION (\d+)", open(HEADER).read()).group(1))
    assert glu.glu_version() == v


def test_status_strings():
    for s in (OK, NULL, SHAPE, STRIDE, ALIAS, ENUM, CUDA):
        assert glu.glu_status_string(s) and glu.glu_status_string(s) != "unknown status"
    assert glu.glu_status_string(12345) == "unknown status"


def fwd(a=BASE, sa=64, b=BASE + (1 << 20), sb=64, y=BASE + (2 << 20), sy=64,
        rows=4, cols=64, layout=SPLIT, act=SILU, dtype=BF16):
    return glu.glu_fwd(a, sa, b, sb, y, sy, rows, cols, layout, act, dtype, None)


def bwd(dc=BASE + (3 << 20), sdc=64, a=BASE, sa=64, b=BASE + (1 << 20), sb=64,
        da=BASE + (4 << 20), sda=64, db=BASE + (5 << 20), sdb=64, rows=4, cols=64,
        layout=SPLIT, act=SILU, dtype=BF16):
    return glu.glu_bwd(dc, sdc, a, sa, b, sb, da, sda, db, sdb, rows, cols, layout, act, dtype, None)


@cpu_only
def test_bad_enums():
    assert fwd(layout=2) == ENUM
    assert fwd(act=4) == ENUM and fwd(act=-1) == ENUM
    assert fwd(dtype=3) == ENUM
    assert bwd(layout=7) == ENUM and bwd(act=9) == ENUM and bwd(dtype=-2) == ENUM


@cpu_only
def test_shapes():
    assert fwd(rows=-1) == SHAPE and fwd(cols=-5) == SHAPE
    assert bwd(rows=-1) == SHAPE
    # byte extent overflow
    assert fwd(rows=1 << 40, sa=1 << 30, sb=1 << 30, sy=1 << 30, cols=1 << 30) == SHAPE


@cpu_only
def test_empty_is_a_noop_even_with_null_pointers():
    assert fwd(a=None, b=None, y=None, rows=0) == OK
    assert fwd(a=None, b=None, y=None, cols=0) == OK
    assert bwd(dc=None, a=None, b=None, da=None, db=None, rows=0) == OK
    assert glu.glu_last_launch()["launched"] == 0


@cpu_only
def test_null_pointers():
    assert fwd(a=None) == NULL and fwd(b=None) == NULL and fwd(y=None) == NULL
    # b is ignored for CONCAT: the call gets past the NULL check and stops at y's stride
    assert fwd(b=None, layout=CONCAT, sa=128, sy=3) == STRIDE
    for k in ("dc", "a", "b", "da", "db"):
        assert bwd(**{k: None}) == NULL, k


@cpu_only
def test_strides():
    assert fwd(sa=63) == STRIDE and fwd(sb=10) == STRIDE and fwd(sy=0) == STRIDE
    assert fwd(sa=-64) == STRIDE
    assert fwd(layout=CONCAT, sa=127) == STRIDE                 # x holds 2 * n_cols per row
    assert bwd(sdc=63) == STRIDE and bwd(sdb=1) == STRIDE
    assert bwd(layout=CONCAT, sa=128, sda=127) == STRIDE


@cpu_only
def test_partial_aliasing_is_rejected():
    # y shifted by one element against b
    assert fwd(y=BASE + (1 << 20) + 2) == ALIAS
    # y == b but with another stride
    assert fwd(b=BASE + (1 << 20), sb=64, y=BASE + (1 << 20), sy=128) == ALIAS
    # y overlapping a by one row
    assert fwd(y=BASE + 64 * 2) == ALIAS
    # two backward outputs overlapping
    assert bwd(da=BASE + (4 << 20), db=BASE + (4 << 20) + 32) == ALIAS
    assert bwd(da=BASE + (4 << 20), db=BASE + (4 << 20)) == ALIAS
    # CONCAT: y over the gate half is a partial overlap of x's rows
    assert fwd(layout=CONCAT, sa=128, y=BASE + 2, sy=128) == ALIAS


@cpu_only
def test_valid_calls_reach_the_cuda_runtime_without_a_gpu():
    """Exact aliasing and interleaved-but-disjoint rows pass validation; with no
    GPU the launch then fails cleanly with GLU_ERR_CUDA and a message."""
    cases = [
        fwd(),                                                   # out of place
        fwd(y=BASE + (1 << 20)),                                 # in place over b
        fwd(y=BASE, sy=64),                                      # in place over a
        fwd(layout=CONCAT, sa=128, b=None, sb=0, y=BASE + 128, sy=128),   # y = x[:, I:]
        fwd(b=BASE + 128, sa=256, sb=256, y=BASE + 256, sy=256),         # rows interleave
        bwd(da=BASE, db=BASE + (1 << 20)),                       # in place backward
        bwd(layout=CONCAT, sa=128, b=None, sb=0, da=BASE, sda=128, db=None, sdb=0),
    ]
    assert cases == [CUDA] * len(cases)
    assert glu.glu_last_cuda_error()


def test_tuning_roundtrip_and_validation():
    glu.glu_set_tuning(16, 4, 8, -1, 2)
    assert glu.glu_get_tuning() == {"vec_bytes": 16, "unroll": 4, "ctas_per_sm": 8, "dependent_launch": -1,
                                    "path": 2}
    for bad in ((8, 0, 0, 0, 0), (0, 3, 0, 0, 0), (0, 0, 100, 0, 0), (0, 0, 0, 2, 0), (0, 0, 0, 0, 3)):
        with pytest.raises(glu.GluError):
            glu.glu_set_tuning(*bad)
    glu.glu_set_tuning(0, 0, 0, 0, 0)
    assert glu.glu_get_tuning() == {"vec_bytes": 0, "unroll": 0, "ctas_per_sm": 0, "dependent_launch": 0,
                                    "path": 0}


def test_last_launch_requires_pointer():
    assert glu.lib().glu_last_launch(None) == NULL


FASTDIV_DRIVER = r"""
#include <cstdio>
#include <cstdint>
#include "glu_plan.h"
int main() {
    const uint32_t ds[] = {1u, 2u, 3u, 7u, 10u, 11u, 250u, 688u, 1376u, 1792u, 2368u, 4096u,
                           65535u, 65536u, 1000003u, 2147483647u, 2147483648u, 2147483649u,
                           4294967295u};
    const uint32_t ns[] = {0u, 1u, 2u, 3u, 99u, 65535u, 65536u, 123456789u, 2147483647u,
                           2147483648u, 3000000000u, 4294967294u, 4294967295u};
    unsigned long long bad = 0, checked = 0;
    for (uint32_t d : ds) {
        uint32_t m, s;
        glu::fastdiv_init(d, &m, &s);
        for (uint32_t n : ns) { ++checked; if (glu::fastdiv(n, m, s) != n / d) ++bad; }
        uint64_t x = 88172645463325252ull;
        for (int i = 0; i < 200000; ++i) {
            x ^= x << 13; x ^= x >> 7; x ^= x << 17;
            uint32_t n = uint32_t(x);
            ++checked; if (glu::fastdiv(n, m, s) != n / d) ++bad;
            uint32_t k = uint32_t(x >> 32) % 4096u;       // exact multiples and neighbours
            uint64_t mult = uint64_t(k) * d;
            if (mult + 1 <= 0xFFFFFFFFull) {
                uint32_t a = uint32_t(mult), b = uint32_t(mult + 1);
                checked += 2;
                if (glu::fastdiv(a, m, s) != a / d) ++bad;
                if (glu::fastdiv(b, m, s) != b / d) ++bad;
                if (a) { ++checked; if (glu::fastdiv(a - 1, m, s) != (a - 1) / d) ++bad; }
            }
        }
    }
    printf("%llu %llu\n", checked, bad);
    return bad != 0;
}
"""


def test_fastdiv_host_logic(tmp_path):
    """The multiply-shift division the kernels use to map a unit index to its
    row, checked against integer division on the host."""
    src = tmp_path / "fd.cpp"
    src.write_text(FASTDIV_DRIVER)
    exe = tmp_path / "fd"
    csrc = os.path.join(ROOT, "glu_activation_mlps_gb300", "csrc")
    cuda_inc = "/usr/local/cuda/include"
    subprocess.run(["g++", "-O2", "-std=c++17", f"-I{csrc}", f"-I{os.path.join(ROOT, 'include')}",
                    f"-I{cuda_inc}", str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    checked, bad = map(int, out.stdout.split())
    assert out.returncode == 0 and bad == 0 and checked > 1_000_000


@cpu_only
def test_host_entry_points_validate_before_any_cuda_call():
    WS = BASE + (8 << 20)
    fh = lambda **k: glu.glu_fwd_host(*[k.get(n, d) for n, d in (
        ("a", BASE), ("sa", 64), ("b", BASE + (1 << 20)), ("sb", 64), ("y", BASE + (2 << 20)), ("sy", 64),
        ("rows", 4), ("cols", 64), ("layout", SPLIT), ("act", SILU), ("dtype", BF16),
        ("ws", WS), ("wsb", 1 << 20), ("s1", None), ("s2", None), ("s3", None))])
    assert fh(rows=0) == OK and fh(act=7) == ENUM and fh(rows=-1) == SHAPE
    assert fh(a=None) == NULL and fh(sy=3) == STRIDE
    assert fh(y=BASE + (1 << 20) + 2) == ALIAS
    assert fh(ws=None) == -7                                  # GLU_ERR_WORKSPACE
    need = glu.glu_host_workspace_bytes(1, 64, SPLIT, BF16, 0)
    assert fh(wsb=need - 1) == -7
    bh = glu.glu_bwd_host(BASE, 64, BASE + (1 << 20), 64, BASE + (2 << 20), 64, BASE + (3 << 20), 64,
                          BASE + (4 << 20), 64, 4, 64, SPLIT, SILU, BF16, WS, 16, None, None, None)
    assert bh == -7


def test_host_workspace_size_formula():
    ws = glu.glu_host_workspace_bytes
    # two slots; each staged matrix rounded up to 256 bytes
    assert ws(1, 64, SPLIT, BF16, 0) == 2 * 3 * 256
    assert ws(100, 1000, SPLIT, BF16, 0) == 2 * 3 * (200192)                  # 100*1000*2 -> 200192
    assert ws(100, 1000, CONCAT, F32, 0) == 2 * (800000 + 400128)             # x (2I) | y
    assert ws(10, 1024, SPLIT, F16, 1) == 2 * 5 * 20480                       # dc, a, b | da, db
    assert ws(10, 1024, CONCAT, F16, 1) == 2 * (20480 + 40960 + 40960)        # dc, x | dx
    assert ws(0, 64, SPLIT, BF16, 0) == 0 and ws(4, 64, 9, BF16, 0) == 0


# ---- glu_gemm_fwd -------------------------------------------------------------

def gemm(x=BASE, sx=64, wg=BASE + (1 << 20), wu=BASE + (2 << 20), sw=64, y=BASE + (3 << 20), sy=96,
         M=4, K=64, I=96, act=SILU, dtype=BF16):
    return glu.glu_gemm_fwd(x, sx, wg, wu, sw, y, sy, M, K, I, act, dtype, None)


@cpu_only
def test_gemm_validation():
    assert gemm(dtype=F32) == ENUM and gemm(dtype=3) == ENUM and gemm(act=4) == ENUM
    assert gemm(M=-1) == SHAPE and gemm(K=-1) == SHAPE and gemm(I=1 << 31) == SHAPE
    assert gemm(x=None, y=None, M=0) == OK and gemm(wg=None, I=0, y=None) == OK
    assert gemm(x=None) == NULL and gemm(wu=None) == NULL and gemm(y=None) == NULL
    assert gemm(sx=63) == STRIDE and gemm(sw=32) == STRIDE and gemm(sy=95) == STRIDE
    # the tensor-memory accelerator's alignment rules: bases and row strides on 16 bytes
    assert gemm(x=BASE + 2) == STRIDE and gemm(wg=BASE + (1 << 20) + 8) == STRIDE
    assert gemm(sx=68) == STRIDE and gemm(sw=66) == STRIDE
    # y over x, over either weight
    assert gemm(y=BASE + 2) == ALIAS
    assert gemm(y=BASE + (2 << 20) + 64 * 2 * 50) == ALIAS
    assert gemm(y=BASE + (1 << 20) - 4) == ALIAS


@cpu_only
def test_gemm_valid_call_reaches_the_cuda_runtime_without_a_gpu():
    # y may be unaligned and strided; the inputs may overlap one another
    assert gemm(y=BASE + (3 << 20) + 2, sy=101) == CUDA
    assert gemm(wu=BASE + (1 << 20)) == CUDA
    assert glu.glu_last_cuda_error()


# ---- glu_gemm_nt and glu_mlp_fwd -------------------------------------------

def gemm_nt(a=BASE, sa=64, b=BASE + (1 << 20), sb=64, d=BASE + (3 << 20), sd=96, M=4, K=64, N=96, dtype=BF16):
    return glu.glu_gemm_nt(a, sa, b, sb, d, sd, M, K, N, dtype, None)


@cpu_only
def test_gemm_nt_validation():
    assert gemm_nt(dtype=F32) == ENUM and gemm_nt(M=-1) == SHAPE and gemm_nt(N=1 << 31) == SHAPE
    assert gemm_nt(a=None, d=None, M=0) == OK and gemm_nt(b=None, N=0, d=None) == OK
    assert gemm_nt(a=None) == NULL and gemm_nt(b=None) == NULL and gemm_nt(d=None) == NULL
    assert gemm_nt(sa=63) == STRIDE and gemm_nt(sb=60) == STRIDE and gemm_nt(sd=95) == STRIDE
    assert gemm_nt(a=BASE + 2) == STRIDE and gemm_nt(sb=66) == STRIDE
    assert gemm_nt(d=BASE + 2) == ALIAS and gemm_nt(d=BASE + (1 << 20) - 4) == ALIAS
    assert gemm_nt(d=BASE + (3 << 20) + 2, sd=101) == CUDA          # valid: reaches the runtime


WS = BASE + (6 << 20)


def mlp(x=BASE, sx=64, wg=BASE + (1 << 20), wu=BASE + (2 << 20), sw=64, wd=BASE + (4 << 20), sd=96,
        out=BASE + (3 << 20), so=64, M=4, H=64, I=96, act=SILU, dtype=BF16, ws=WS, ws_bytes=1 << 20):
    return glu.glu_mlp_fwd(x, sx, wg, wu, sw, wd, sd, out, so, M, H, I, act, dtype, ws, ws_bytes, None)


@cpu_only
def test_mlp_validation():
    assert mlp(act=4) == ENUM and mlp(dtype=F32) == ENUM
    assert mlp(M=-1) == SHAPE and mlp(I=-1) == SHAPE and mlp(H=1 << 31) == SHAPE
    assert mlp(x=None, out=None, M=0) == OK and mlp(x=None, out=None, H=0) == OK
    assert mlp(x=None) == NULL and mlp(wd=None) == NULL and mlp(out=None) == NULL
    assert mlp(sx=63) == STRIDE and mlp(sw=63) == STRIDE and mlp(so=60) == STRIDE and mlp(sd=95) == STRIDE
    # the workspace holds at least one row of y (I rounded up to 8 elements)
    assert mlp(ws=None) == WORKSPACE and mlp(ws_bytes=2 * 96 - 2) == WORKSPACE
    assert mlp(I=97, sd=104, ws_bytes=2 * 97) == WORKSPACE and mlp(I=97, sd=104, ws_bytes=2 * 104) == CUDA
    # the tensor-memory accelerator's alignment rules, before any launch
    assert mlp(ws=WS + 8) == STRIDE and mlp(wd=BASE + (4 << 20) + 2) == STRIDE and mlp(sd=100) == STRIDE
    # out may overlap nothing: not x, a weight or the workspace
    assert mlp(out=BASE) == ALIAS and mlp(out=BASE + (4 << 20) + 64) == ALIAS and mlp(out=WS + 512) == ALIAS
    assert mlp() == CUDA and glu.glu_last_cuda_error()              # valid: reaches the runtime


def test_mlp_workspace_bytes():
    ws = glu.glu_mlp_workspace_bytes
    assert ws(4096, 14336, BF16) == 4096 * 14336 * 2          # the whole y
    assert ws(65536, 14336, BF16) == 37376 * 14336 * 2        # 1 GiB holds 37449 rows: 146 blocks of 256
    assert ws(100, 14336, BF16) == 100 * 14336 * 2 and ws(10, 97, F16) == 10 * 104 * 2
    assert ws(0, 64, BF16) == 0 and ws(4, 64, F32) == 0 and ws(4, 0, BF16) == 0


# ---- glu_add_rmsnorm_fwd -----------------------------------------------------

VALUE = -8


def rms(x=BASE, sx=64, r=BASE + (1 << 20), sr=64, g=BASE + (2 << 20), h=BASE + (3 << 20), sh=64,
        y=BASE + (4 << 20), sy=64, rstd=BASE + (5 << 20), rows=4, cols=64, eps=1e-5, dtype=BF16):
    return glu.glu_add_rmsnorm_fwd(x, sx, r, sr, g, h, sh, y, sy, rstd, rows, cols, eps, dtype, None)


@cpu_only
def test_add_rmsnorm_validation():
    assert rms(dtype=3) == ENUM and rms(dtype=-1) == ENUM
    assert rms(rows=-1) == SHAPE and rms(cols=-2) == SHAPE
    assert rms(cols=32769, sx=40000, sr=40000, sh=40000, sy=40000) == SHAPE
    for bad in (0.0, -1e-5, float("nan"), float("inf")):
        assert rms(eps=bad) == VALUE, bad
    assert rms(x=None, r=None, g=None, h=None, y=None, rstd=None, rows=0) == OK
    for k in ("x", "r", "g", "h", "y"):
        assert rms(**{k: None}) == NULL, k
    assert rms(sx=63) == STRIDE and rms(sh=10) == STRIDE and rms(sy=0) == STRIDE
    # outputs: exactly an input is fine (checked with a GPU); any other overlap is not
    assert rms(h=BASE + 2) == ALIAS                                 # h one element past x
    assert rms(h=BASE + (3 << 20), y=BASE + (3 << 20) + 64) == ALIAS   # h and y overlap
    assert rms(h=BASE, y=BASE) == ALIAS                             # both over x
    assert rms(y=BASE + (2 << 20) + 6) == ALIAS                     # y over gamma
    assert rms(rstd=BASE + 8) == ALIAS and rms(rstd=BASE + (4 << 20) + 100) == ALIAS
    assert glu.glu_status_string(VALUE) != "unknown status"


@cpu_only
def test_add_rmsnorm_valid_calls_reach_the_cuda_runtime_without_a_gpu():
    assert rms() == CUDA                                  # out of place
    assert rms(h=BASE, y=BASE + (1 << 20)) == CUDA        # h over x, y over the residual
    assert rms(h=BASE + (1 << 20), y=BASE, rstd=None) == CUDA
    assert rms(x=BASE + 2, sx=67, cols=61) == CUDA        # unaligned: element accesses


def rmsb(dy=BASE, sdy=64, h=BASE + (1 << 20), sh=64, rstd=BASE + (2 << 20), g=BASE + (3 << 20),
         dh=None, sdh=0, dx=BASE + (4 << 20), sdx=64, dres=None, sdr=0, dg=BASE + (5 << 20), rows=4, cols=64,
         dtype=BF16):
    return glu.glu_add_rmsnorm_bwd(dy, sdy, h, sh, rstd, g, dh, sdh, dx, sdx, dres, sdr, dg, rows, cols, dtype, None)


@cpu_only
def test_add_rmsnorm_bwd_validation():
    assert rmsb(dtype=5) == ENUM
    assert rmsb(rows=-1) == SHAPE and rmsb(cols=16385, sdy=16400, sh=16400, sdx=16400) == SHAPE
    assert rmsb(dy=None, h=None, rstd=None, g=None, dx=None, dg=None, rows=0) == OK
    for k in ("dy", "h", "rstd", "g", "dx"):
        assert rmsb(**{k: None}) == NULL, k
    assert rmsb(sdy=63) == STRIDE and rmsb(sdx=1) == STRIDE
    assert rmsb(dh=BASE + (6 << 20), sdh=3) == STRIDE and rmsb(dres=BASE + (7 << 20), sdr=5) == STRIDE
    assert rmsb(dx=BASE + 4) == ALIAS                                     # dx shifted over dy
    assert rmsb(dres=BASE + (4 << 20), sdr=64) == ALIAS                   # dres on dx
    assert rmsb(dx=BASE + (3 << 20) + 2) == ALIAS                         # dx over gamma
    assert rmsb(dx=BASE + (2 << 20)) == ALIAS                             # dx over rstd
    assert rmsb(dg=BASE + 100) == ALIAS and rmsb(dg=BASE + (3 << 20) + 4) == ALIAS
    assert rmsb(dg=BASE + (2 << 20) + 8) == ALIAS                         # dgamma over rstd


@cpu_only
def test_add_rmsnorm_bwd_valid_calls_reach_the_cuda_runtime_without_a_gpu():
    assert rmsb() == CUDA
    assert rmsb(dx=BASE, dres=BASE + (1 << 20), sdr=64, dg=None) == CUDA      # in place over dy and h
    assert rmsb(dh=BASE + (6 << 20), sdh=64, dx=BASE + (6 << 20)) == CUDA    # in place over dh
