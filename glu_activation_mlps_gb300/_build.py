"""In-tree build of the CUDA library ``libglu_gb300.so`` for sm_103a.

Each translation unit is compiled by its own nvcc process (in parallel), then
linked into one shared library with the CUDA runtime linked statically.  No
fast-math and no flush-to-zero: subnormal results are part of the numerical
contract.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libglu_gb300.so")

SOURCES = ["glu_api.cu", "glu_host.cu", "glu_noalloc.cu", "glu_bulk.cu", "glu_inst_bf16.cu",
           "glu_inst_f16.cu", "glu_inst_f32.cu", "glu_gemm.cu", "glu_rmsnorm.cu"]
HEADERS = ["glu_plan.h", "glu_internal.h", "glu_math.cuh", "glu_kernels.cuh", "glu_bulk.cuh", "glu_async.cuh"]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo", "-O3", "-std=c++17",
    "-Xcompiler", "-fPIC",
    "-I" + INCLUDE, "-I" + CSRC,
]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the library")
    return cand


def _inputs():
    deps = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "glu.h"), __file__]
    return deps


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    common = _inputs()
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, common + [s]):
            jobs.append([nvcc(), *NVCC_FLAGS, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        if verbose:
            sys.stdout.write(r.stdout + r.stderr)

    if jobs:
        with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            list(ex.map(run, jobs))
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        run([nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared",
             "-Xcompiler", "-fPIC", "-o", tmp, *objs])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
