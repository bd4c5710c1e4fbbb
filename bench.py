"""Benchmark of the fused gated activation on GB300.

One step = the whole hot path over one batch: the SwiGLU forward
y = silu(a) * b and the backward (da, db) = (dc * silu'(a) * b, dc * silu(a))
on bf16 matrices of 4096 x 14336 (4096 tokens at intermediate size 14336),
through the C ABI (glu_fwd, glu_bwd).  The metric is achieved HBM bandwidth:
algorithmic bytes (forward 3 x 2 B, backward 5 x 2 B per element) over time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun every rank runs its own batch on its own GPU (weak scaling, no
data-path collective); rank 0 prints one JSON line.  `--impl reference` times
the double-precision CPU oracle on the host cores instead (the only other
implementation of this computation), on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import glu_synth  # noqa: E402

ROWS, COLS = 4096, 14336
E = 2
N_ELEMS = ROWS * COLS
FWD_BYTES = 3 * E * N_ELEMS
BWD_BYTES = 5 * E * N_ELEMS
STEP_BYTES = FWD_BYTES + BWD_BYTES
METRIC = "SwiGLU fwd+bwd achieved HBM GB/s (% of GB300 peak), bf16 BT=4096 I=14336"
UNIT = "GB/s"
WORKLOAD = "swiglu_fwd_bwd_bf16_4096x14336"
L2_BYTES = 126 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
CSRC = os.path.join(ROOT, "glu_activation_mlps_gb300", "csrc")


def config(extra=None):
    c = {"workload": WORKLOAD, "act": "silu", "layout": "split", "n_rows": ROWS, "n_cols": COLS,
         "storage": "bf16", "math": "f32", "backward": "out-of-place (da, db separate)",
         "l2": f"no flush: inputs larger than L2 ({STEP_BYTES / 1e6:.0f} MB touched per step, "
               f"{FWD_BYTES / 1e6:.0f} MB per forward, vs {L2_BYTES / 2**20:.0f} MiB L2)",
         "inputs": "seeded synthetic a, b, dc ~ N(0, 1)"}
    if extra:
        c.update(extra)
    return c


# the sources the streaming kernels are compiled from; their launch shape is
# compared separately (ncu_traffic)
STREAMING_SOURCES = ("glu_inst_bf16.cu", "glu_kernels.cuh", "glu_math.cuh", "glu_plan.h")
LAUNCH_KEYS = ("vec_bytes", "unroll", "threads", "grid", "flattened", "path")


def source_sha() -> str:
    h = hashlib.sha256()
    for f in STREAMING_SOURCES:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def ncu_traffic(launch_bwd=None):
    """Per-launch DRAM bytes of the backward kernel from the committed ncu
    summary, or None if the kernel sources or its launch shape changed since
    it was taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("source_sha") != source_sha():
        return None
    rec = t.get("bwd_launch")
    if launch_bwd is not None and rec is not None and any(rec.get(k) != launch_bwd.get(k) for k in LAUNCH_KEYS):
        return None
    return t.get("bwd_dram_bytes_per_launch")


# ---------------------------------------------------------------- ranks

def reduce_max(x: float, device=None) -> float:
    """Max of `x` over all ranks (the job's time is its slowest rank's); the
    value itself when no process group is running.  Only timings travel: the
    ranks exchange no data of the computation."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def link_ceiling(src_host, dst_host, dev_buf, s_a, s_b, reps=5):
    """GB/s of cudaMemcpyAsync between pinned host memory and the device:
    host->device, device->host, and both at once on two streams (the bytes of
    both directions over the time of the pair)."""
    import torch
    nbytes = min(src_host.numel() * src_host.element_size(), dst_host.numel() * dst_host.element_size(),
                 dev_buf.numel() * dev_buf.element_size() // 2)
    hs = src_host.view(-1).view(torch.uint8)[:nbytes]
    hd = dst_host.view(-1).view(torch.uint8)[:nbytes]
    d0, d1 = dev_buf.view(torch.uint8)[:nbytes], dev_buf.view(torch.uint8)[nbytes:2 * nbytes]
    cur = torch.cuda.current_stream()

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        for _ in range(reps):
            fn()
        b.record(cur)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    def both():
        s_a.wait_stream(cur)
        s_b.wait_stream(cur)
        with torch.cuda.stream(s_a):
            d0.copy_(hs, non_blocking=True)
        with torch.cuda.stream(s_b):
            hd.copy_(d1, non_blocking=True)
        cur.wait_stream(s_a)
        cur.wait_stream(s_b)

    h2d = timed(lambda: d0.copy_(hs, non_blocking=True))
    d2h = timed(lambda: hd.copy_(d1, non_blocking=True))
    bi = timed(both)
    return {"h2d_gbs": round(nbytes / h2d / 1e6, 1), "d2h_gbs": round(nbytes / d2h / 1e6, 1),
            "both_gbs": round(2 * nbytes / bi / 1e6, 1), "bytes": nbytes,
            "method": "cudaMemcpyAsync by the copy engines on the same pinned buffers; both directions at "
                      "once on two streams"}


def job_gbs(world: int, steps: int, bytes_per_step: int, ms: float) -> float:
    """Whole-job throughput: every rank runs its own batch (weak scaling), so
    the job moves world * steps * bytes_per_step in the slowest rank's time."""
    return world * steps * bytes_per_step / (ms * 1e-3) / 1e9


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: str):
        self.samples = []
        self.proc = None
        self.idx = device
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.idx)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        deadline = time.time() + 5
        while not self.samples and time.time() < deadline:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self, start: bool):
        if start:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [s for t, s in self.samples if self.t0 - 0.06 <= t <= self.t1 + 0.06]
        if not rows:
            rows = [s for _, s in self.samples][-3:]
        try:
            sm = [float(r[1]) for r in rows]
            smax = max(float(r[2]) for r in rows)
        except (ValueError, IndexError):
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if len(r) > 5 + i and r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows)}


def gpu_selector(local_rank: int) -> str:
    """nvidia-smi's id for this process's CUDA device (its UUID when known:
    CUDA ordinals and nvidia-smi indices differ under CUDA_VISIBLE_DEVICES)."""
    try:
        import torch
        u = str(torch.cuda.get_device_properties(local_rank).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        parts = [p for p in vis.split(",") if p.strip()]
        return parts[local_rank].strip() if local_rank < len(parts) else str(local_rank)


# ---------------------------------------------------------------- GPU arm

def run_gpu(args, rank, world, local_rank):
    import torch
    import glu_activation_mlps_gb300 as glu
    from glu_activation_mlps_gb300 import ACT, DTYPE, LAYOUT

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if local_rank == 0:
        glu.build()
    if world > 1:
        torch.distributed.barrier()
    glu.lib()
    glu.glu_set_tuning(path={"default": 0, "direct": 1, "bulk": 2}[args.path])

    d = glu_synth.metric_bf16()
    host = {k: torch.from_numpy(d[k].view(np.int16)).pin_memory() for k in ("a", "b", "dc")}
    A, B, DC = (host[k].to(dev).view(torch.bfloat16) for k in ("a", "b", "dc"))
    Y, DA, DB = (torch.empty_like(A) for _ in range(3))
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    silu, split, bf16 = ACT["silu"], LAYOUT["split"], DTYPE["bf16"]
    L = glu.lib()
    pa, pb, pc, py, pda, pdb = (t.data_ptr() for t in (A, B, DC, Y, DA, DB))

    def fwd():
        st = L.glu_fwd(pa, COLS, pb, COLS, py, COLS, ROWS, COLS, split, silu, bf16, sh)
        if st:
            raise glu.GluError(st, "glu_fwd")

    def bwd():
        st = L.glu_bwd(pc, COLS, pa, COLS, pb, COLS, pda, COLS, pdb, COLS, ROWS, COLS, split, silu, bf16, sh)
        if st:
            raise glu.GluError(st, "glu_bwd")

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        fwd()
        launch_fwd = dict(glu.glu_last_launch())
        bwd()
        launch_bwd = dict(glu.glu_last_launch())
    torch.cuda.synchronize()

    clocks = ClockSampler(gpu_selector(local_rank)) if rank == 0 else None
    if clocks:
        clocks.start()
    K = args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.mark(True)
    # the timed region: exactly K steps, nothing else enqueued between kernels
    start.record(stream)
    for k in range(K):
        fwd()
        bwd()
    end.record(stream)
    torch.cuda.synchronize()
    if clocks:
        clocks.mark(False)
    barrier()
    total_ms = start.elapsed_time(end)
    launches = 2 * K    # the headline region; the event pass and the e2e runs follow it
    clock_info = clocks.stop() if clocks else None

    # per-kernel durations for the roofline: the same K steps again, with an
    # event pair around every launch on the launching stream (events between
    # kernels break the launch overlap, so this pass is not the headline)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    barrier()
    torch.cuda.synchronize()
    for k in range(K):
        ev[k][0].record(stream)
        fwd()
        ev[k][1].record(stream)
        bwd()
        ev[k][2].record(stream)
    torch.cuda.synchronize()
    barrier()
    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in ev]

    total_ms = reduce_max(total_ms, dev)

    # end to end through the C ABI's host-memory entry points: a, b, dc live in
    # page-locked host memory; each step's glu_fwd_host copies a, b in and y
    # out, glu_bwd_host copies dc, a, b in and da, db out, overlapping the
    # copies with the kernels through a 128 MiB device workspace
    out_host = {k: torch.empty_like(host["a"]).pin_memory() for k in ("y", "da", "db")}
    ws_bytes = 128 << 20
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    hp = {k: host[k].data_ptr() for k in ("a", "b", "dc")}
    op = {k: out_host[k].data_ptr() for k in out_host}
    Ke = max(3, min(K, 20))

    def e2e_step():
        st = L.glu_fwd_host(hp["a"], COLS, hp["b"], COLS, op["y"], COLS, ROWS, COLS, split, silu, bf16,
                            ws.data_ptr(), ws_bytes, s_in.cuda_stream, sh, s_out.cuda_stream)
        if st:
            raise glu.GluError(st, "glu_fwd_host")
        st = L.glu_bwd_host(hp["dc"], COLS, hp["a"], COLS, hp["b"], COLS, op["da"], COLS, op["db"], COLS,
                            ROWS, COLS, split, silu, bf16, ws.data_ptr(), ws_bytes, s_in.cuda_stream, sh,
                            s_out.cuda_stream)
        if st:
            raise glu.GluError(st, "glu_bwd_host")

    for _ in range(2):
        e2e_step()
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(Ke):
        e2e_step()
    e1.record(stream)          # the compute stream waits for each call's last copy out
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1), dev)
    barrier()

    # the same step with the device entry points on the pinned host buffers
    # themselves: the kernels read a, b, dc from host memory and write y, da,
    # db back over the host link (zero-copy; every byte still crosses the link
    # inside the timed region)
    def zc_step():
        st = L.glu_fwd(hp["a"], COLS, hp["b"], COLS, op["y"], COLS, ROWS, COLS, split, silu, bf16, sh)
        if st:
            raise glu.GluError(st, "glu_fwd")
        st = L.glu_bwd(hp["dc"], COLS, hp["a"], COLS, hp["b"], COLS, op["da"], COLS, op["db"], COLS, ROWS, COLS,
                       split, silu, bf16, sh)
        if st:
            raise glu.GluError(st, "glu_bwd")

    for _ in range(2):
        zc_step()
    barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(Ke):
        zc_step()
    e1.record(stream)
    torch.cuda.synchronize()
    zc_ms = reduce_max(e0.elapsed_time(e1), dev)
    barrier()

    # the host link's own ceiling for the e2e number: the copy engines moving
    # the same pinned bytes one way, the other way, and both ways at once
    link = link_ceiling(host["a"], out_host["y"], ws, s_in, s_out)
    barrier()

    if rank != 0:
        return None

    peak, peak_src = measured_peak()
    bwd_avg = statistics.fmean(bwd_ms)
    fwd_avg = statistics.fmean(fwd_ms)
    achieved = BWD_BYTES / (bwd_avg * 1e-3) / 1e9
    traffic = ncu_traffic(launch_bwd)
    value = job_gbs(world, K, STEP_BYTES, total_ms)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(total_ms / K, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config({"parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                          "launch": {"fwd": launch_fwd, "bwd": launch_bwd}}),
        "roofline": {"bound": "hbm", "kernel": "backward (glu_bwd)", "achieved": round(achieved, 1),
                     "peak": peak, "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, copy)",
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic, "algorithmic_bytes": BWD_BYTES},
        "per_kernel": {"fwd_ms": round(fwd_avg, 5), "bwd_ms": round(bwd_avg, 5),
                       "fwd_gbs": round(FWD_BYTES / (fwd_avg * 1e-3) / 1e9, 1),
                       "bwd_gbs": round(achieved, 1),
                       "fwd_frac": round(FWD_BYTES / (fwd_avg * 1e-3) / 1e9 / peak, 4),
                       "fwd_min_ms": round(min(fwd_ms), 5), "bwd_min_ms": round(min(bwd_ms), 5)},
        "e2e": {"value": round(job_gbs(world, Ke, STEP_BYTES, zc_ms), 1), "unit": UNIT,
                "h2d_bytes_per_step": 5 * E * N_ELEMS, "d2h_bytes_per_step": 3 * E * N_ELEMS,
                "steps": Ke, "ms_per_step": round(zc_ms / Ke, 4),
                "api": "glu_fwd + glu_bwd on pinned host buffers: the kernels read and write host memory "
                       "in place over the host link (zero-copy)",
                "link": link,
                "frac_of_link": round(job_gbs(world, Ke, STEP_BYTES, zc_ms) / world / link["both_gbs"], 4)},
        "e2e_staged": {"value": round(job_gbs(world, Ke, STEP_BYTES, e2e_ms), 1), "unit": UNIT,
                       "h2d_bytes_per_step": 5 * E * N_ELEMS, "d2h_bytes_per_step": 3 * E * N_ELEMS,
                       "steps": Ke, "ms_per_step": round(e2e_ms / Ke, 4),
                       "api": "glu_fwd_host + glu_bwd_host (pinned host buffers copied through a 128 MiB "
                              "device workspace by the copy engines)"},
        "gpu_launches": launches,
        "roofline_pass": f"per-kernel CUDA events over a second pass of {K} steps ({2 * K} launches)",
        "tuning": glu.glu_get_tuning(),
        "clocks": clock_info,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(d, budget_s=args.cpu_seconds)
    return line


# ---------------------------------------------------------------- throughput table

def run_table(args):
    """Throughput of every named workload with the library defaults (or the
    --path given): back-to-back launches over rotating sets of buffers whose
    total exceeds L2, median of rounds, against the measured copy bandwidth.
    Prints a markdown table (not the benchmark's JSON line)."""
    import torch
    import glu_activation_mlps_gb300 as glu

    glu.build()
    L = glu.lib()
    glu.glu_set_tuning(path={"default": 0, "direct": 1, "bulk": 2}[args.path])
    peak, src = measured_peak()
    s = torch.cuda.current_stream().cuda_stream
    TD = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
    EB = {"bf16": 2, "f16": 2, "f32": 4}
    code = {"bf16": 2, "f16": 1, "f32": 0}
    gen = torch.Generator(device="cuda").manual_seed(0)

    def sets_for(nbytes_per_set, make):
        n = max(2, -(-600 * 2**20 // nbytes_per_set))
        return [make() for _ in range(n)]

    def timed(fn, nsets, reps=40, rounds=5):
        out = []
        for _ in range(rounds):
            for k in range(5):
                fn(k % nsets)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record()
            for k in range(reps):
                fn(k % nsets)
            e1.record()
            torch.cuda.synchronize()
            out.append(e0.elapsed_time(e1) / reps * 1e3)
        return statistics.median(out)

    rows = []

    def split_case(name, R, C, dt, act, direction, sigma=1.0):
        E_ = EB[dt]

        def make():
            t = [(torch.randn(R, C, device="cuda", generator=gen) * sigma).to(TD[dt]) for _ in range(3)]
            return t + [torch.empty_like(t[0]) for _ in range(2)]
        sets = sets_for(5 * R * C * E_, make)
        a_ = glu.ACT[act]

        def fn(k):
            A, B, DC, Y0, Y1 = sets[k]
            if direction == "fwd":
                st = L.glu_fwd(A.data_ptr(), C, B.data_ptr(), C, Y0.data_ptr(), C, R, C, 0, a_, code[dt], s)
            else:
                st = L.glu_bwd(DC.data_ptr(), C, A.data_ptr(), C, B.data_ptr(), C, Y0.data_ptr(), C,
                               Y1.data_ptr(), C, R, C, 0, a_, code[dt], s)
            assert st == 0
        us = timed(fn, len(sets))
        nb = (3 if direction == "fwd" else 5) * E_ * R * C
        rows.append((name, f"{R}x{C}", dt, act, direction, us, nb / us / 1e3))

    def concat_case(name, R, C, inplace):
        def make():
            x = (torch.randn(R, 2 * C, device="cuda", generator=gen) * 1.5).to(torch.bfloat16)
            return [x, torch.empty(R, C, dtype=torch.bfloat16, device="cuda")]
        sets = sets_for(3 * R * C * 2, make)

        def fn(k):
            X, Y = sets[k]
            y, ys = (X[:, C:], 2 * C) if inplace else (Y, C)
            st = L.glu_fwd(X.data_ptr(), 2 * C, None, 0, y.data_ptr(), ys, R, C, 1, 0, 2, s)
            assert st == 0
        us = timed(fn, len(sets))
        rows.append((name, f"{R}x(2x{C})", "bf16", "silu", "fwd", us, 6 * R * C / us / 1e3))

    split_case("fwd f32 small", 256, 1024, "f32", "silu", "fwd")
    split_case("fwd bf16", 4096, 11008, "bf16", "silu", "fwd", sigma=2.0)
    concat_case("fwd bf16 [gate|up]", 4096, 18944, False)
    concat_case("fwd bf16 [gate|up] in place", 4096, 18944, True)
    split_case("bwd bf16 (in-place shape)", 4096, 28672, "bf16", "silu", "bwd", sigma=3.0)
    split_case("metric fwd", ROWS, COLS, "bf16", "silu", "fwd")
    split_case("metric bwd", ROWS, COLS, "bf16", "silu", "bwd")
    for dt in glu_synth.SWEEP_DTYPES:
        for H in glu_synth.SWEEP_H:
            for act in glu_synth.SWEEP_ACTS:
                for d in ("fwd", "bwd"):
                    split_case("sweep", 4096, H, dt, act, d)
    # context: the same forward and backward as plain PyTorch (eager, and
    # torch.compile where it works on this machine) at the metric shape
    cmp = []
    A = torch.randn(ROWS, COLS, device="cuda", generator=gen).to(torch.bfloat16)
    B = torch.randn(ROWS, COLS, device="cuda", generator=gen).to(torch.bfloat16)
    DC = torch.randn(ROWS, COLS, device="cuda", generator=gen).to(torch.bfloat16)

    def t_fwd(a, b):
        return torch.nn.functional.silu(a.float()).mul(b.float()).to(a.dtype)

    def t_bwd(dc, a, b):
        af, bf, cf = a.float(), b.float(), dc.float()
        sg = torch.sigmoid(af)
        silu = af * sg
        return (cf * (silu * (1 - sg) + sg) * bf).to(a.dtype), (cf * silu).to(a.dtype)

    def once(fn, reps=20):
        for _ in range(3):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps * 1e3

    Y0, Y1 = torch.empty_like(A), torch.empty_like(A)

    def ours_fwd():
        assert L.glu_fwd(A.data_ptr(), COLS, B.data_ptr(), COLS, Y0.data_ptr(), COLS, ROWS, COLS, 0, 0, 2, s) == 0

    def ours_bwd():
        assert L.glu_bwd(DC.data_ptr(), COLS, A.data_ptr(), COLS, B.data_ptr(), COLS, Y0.data_ptr(), COLS,
                         Y1.data_ptr(), COLS, ROWS, COLS, 0, 0, 2, s) == 0

    cmp.append(("fwd", once(ours_fwd), once(lambda: t_fwd(A, B))))
    cmp.append(("bwd", once(ours_bwd), once(lambda: t_bwd(DC, A, B))))
    try:
        cf, cb = torch.compile(t_fwd), torch.compile(t_bwd)
        compiled = [once(lambda: cf(A, B)), once(lambda: cb(DC, A, B))]
    except Exception as exc:       # no compiler toolchain on the GPU machine: report why
        compiled = [f"unavailable ({type(exc).__name__})"] * 2
    print("| SwiGLU bf16 4096x14336 | this library (us) | torch eager (us) | torch.compile (us) |")
    print("|---|---|---|---|")
    for (d, ours, eager), comp in zip(cmp, compiled):
        comp_s = f"{comp:.1f}" if isinstance(comp, float) else comp
        print(f"| {d} | {ours:.1f} | {eager:.1f} | {comp_s} |", flush=True)
    print()
    print(f"| workload | shape | dtype | act | dir | us / launch | GB/s | % of {peak:.0f} GB/s ({src}) |")
    print("|---|---|---|---|---|---|---|---|")
    for name, shape, dt, act, d, us, gbs in rows:
        print(f"| {name} | {shape} | {dt} | {act} | {d} | {us:.2f} | {gbs:.0f} | {100 * gbs / peak:.1f} |",
              flush=True)


# ---------------------------------------------------------------- one workload at a time (ncu captures)

CASES = {
    # name: (generator, dir, act, layout, in place, description)
    "c1": ("fwd_f32_small", "fwd", "silu", "split", False, "SwiGLU fwd f32 256x1024"),
    "c2": ("fwd_bf16_split", "fwd", "silu", "split", False, "SwiGLU fwd bf16 4096x11008"),
    "c3": ("fwd_bf16_concat", "fwd", "silu", "concat", False, "SwiGLU fwd bf16 [gate|up] 4096x(2x18944)"),
    "c3_inplace": ("fwd_bf16_concat", "fwd", "silu", "concat", True,
                   "SwiGLU fwd bf16 [gate|up] 4096x(2x18944), y over the up half"),
    "c4": ("bwd_bf16_outliers", "bwd", "silu", "split", True, "SwiGLU bwd bf16 4096x28672, da->a, db->b"),
    "metric_fwd": ("metric_bf16", "fwd", "silu", "split", False, "SwiGLU fwd bf16 4096x14336"),
    "metric_bwd": ("metric_bf16", "bwd", "silu", "split", False, "SwiGLU bwd bf16 4096x14336"),
    "metric_step": ("metric_bf16", "step", "silu", "split", False,
                    "SwiGLU fwd + bwd bf16 4096x14336 (one benchmark step: two launches)"),
}


def case_data(name):
    """Inputs (host bit arrays) and the call's description for a named
    workload, or for `sweep:<act>:<dtype>:<fwd|bwd>:<H>` (a 4096 x H case of
    the activation sweep)."""
    if name.startswith("sweep:"):
        _, act, dt, direction, H = name.split(":")
        d = glu_synth.sweep(int(H), dt, with_dc=direction == "bwd")
        return d, direction, act, "split", False, f"{act} {direction} {dt} 4096x{H}"
    if name not in CASES:
        raise SystemExit(f"unknown case {name!r}: one of {', '.join(CASES)} or sweep:<act>:<dtype>:<dir>:<H>")
    gen, direction, act, layout, inplace, desc = CASES[name]
    return getattr(glu_synth, gen)(), direction, act, layout, inplace, desc


def run_case(args):
    """One named workload launched --warmup + --steps times, each launch timed
    with CUDA events on its stream; in-place cases restore their inputs before
    every launch, outside the timed pair.  This is the command the per-config
    ncu captures profile (`-k regex:glu_kernel -s <warmup> -c 1`).

    With --graph N the N launches of one repetition (2 N for metric_step) are
    captured into a CUDA graph and the graph is replayed --warmup + --steps
    times: the sustained form, back to back with the launch overlap, that
    `ncu --graph-profiling graph -s <warmup> -c 1` measures as one workload.
    In-place cases then run without restores (each launch works on the
    previous one's output; the arithmetic per element is the same).
    Prints one JSON line (not the benchmark's line)."""
    import torch
    import glu_activation_mlps_gb300 as glu

    glu.build()
    L = glu.lib()
    glu.glu_set_tuning(path={"default": 0, "direct": 1, "bulk": 2}[args.path])
    d, direction, act, layout, inplace, desc = case_data(args.case)
    dt = d["dtype"]
    E_ = glu_synth.ELEM_BYTES[dt]
    code, a_ = glu.DTYPE[dt], glu.ACT[act]
    dev = torch.device("cuda", 0)

    def put(x):
        return torch.from_numpy(x.view(np.int32 if x.dtype == np.uint32 else np.int16)).to(dev)

    keep = []          # (live tensor, pristine copy) pairs restored before each launch
    launches = []      # functions of the stream handle, one kernel launch each
    if layout == "concat":
        X = put(d["x"])
        R, C = X.shape[0], d["n_cols"]
        Y = X[:, C:] if inplace else torch.empty(R, C, dtype=X.dtype, device=dev)
        ys = 2 * C if inplace else C
        if inplace:
            keep.append((X, X.clone()))
        launches.append(lambda sh: L.glu_fwd(X.data_ptr(), 2 * C, None, 0, Y.data_ptr(), ys, R, C,
                                             glu.LAYOUT["concat"], a_, code, sh))
    else:
        A, B = put(d["a"]), put(d["b"])
        R, C = A.shape
        if direction in ("fwd", "step"):
            Y = torch.empty_like(A)
            launches.append(lambda sh: L.glu_fwd(A.data_ptr(), C, B.data_ptr(), C, Y.data_ptr(), C, R, C, 0, a_,
                                                 code, sh))
        if direction in ("bwd", "step"):
            DC = put(d["dc"])
            DA, DB = (A, B) if inplace else (torch.empty_like(A), torch.empty_like(B))
            if inplace:
                keep += [(A, A.clone()), (B, B.clone())]
            launches.append(lambda sh: L.glu_bwd(DC.data_ptr(), C, A.data_ptr(), C, B.data_ptr(), C, DA.data_ptr(),
                                                 C, DB.data_ptr(), C, R, C, 0, a_, code, sh))
    del d
    per_unit = {"fwd": 3, "bwd": 5, "step": 8}[direction]
    nbytes = per_unit * E_ * R * C

    def run_once(sh):
        for fn in launches:
            st = fn(sh)
            if st:
                raise glu.GluError(st, "case launch")

    stream = torch.cuda.current_stream(dev)
    graph = None
    reps = 1
    if args.graph:
        reps = args.graph
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            run_once(side.cuda_stream)           # once outside the capture
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            for _ in range(reps):
                run_once(side.cuda_stream)
        torch.cuda.synchronize()
    times = []
    info = None
    for k in range(args.warmup + args.steps):
        if graph is None:
            for live, pristine in keep:
                live.copy_(pristine)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if graph is None:
            run_once(stream.cuda_stream)
            info = dict(glu.glu_last_launch())
        else:
            graph.replay()
        e1.record(stream)
        if k >= args.warmup:
            times.append((e0, e1))
    torch.cuda.synchronize()
    us = [a.elapsed_time(b) * 1e3 / reps for a, b in times]
    peak, src = measured_peak()
    med = statistics.median(us)
    print(json.dumps({"case": args.case, "what": desc, "rows": R, "cols": C, "dtype": dt, "act": act,
                      "dir": direction, "in_place": inplace, "algorithmic_bytes": nbytes,
                      "graph_reps": reps if graph is not None else None,
                      "launches": (args.warmup + args.steps) * reps * len(launches), "timed": len(us),
                      "us_median": round(med, 3), "us_min": round(min(us), 3),
                      "gbs": round(nbytes / med / 1e3, 1), "frac_of_copy": round(nbytes / med / 1e3 / peak, 4),
                      "peak_source": src, "launch": info}), flush=True)


# ---------------------------------------------------------------- gate/up GEMM with the activation in the epilogue

GM, GK, GI = 4096, 4096, 14336      # tokens, hidden size, intermediate size of one MLP layer


# Other layer shapes for --gemm: token counts from decode (1, 64, 128) to a
# large batch (8192), and a wider layer (hidden 8192, intermediate 28672).
GEMM_SHAPES = ((8192, 4096, 14336), (2048, 4096, 14336), (1024, 4096, 14336), (4096, 8192, 28672),
               (128, 8192, 28672), (64, 4096, 14336), (1, 8192, 28672))


def tile_columns(M, I, info):
    """The column-tile width a glu_gemm_fwd launch used, from its tile count."""
    m_blocks = -(-M // (128 * info["unroll"]))
    i_blocks = info["vector_units"] // m_blocks
    return next(bn for bn in (64, 96, 128) if -(-I // bn) == i_blocks)


def gemm_shapes(L, glu, timed, dev, s, K, W):
    """glu_gemm_fwd against cuBLAS alone and cuBLAS then glu_fwd, per shape."""
    import torch
    out = []
    for (M, Kd, I) in GEMM_SHAPES:
        gen = torch.Generator(device=dev).manual_seed(7)
        x = torch.randn(M, Kd, device=dev, generator=gen).to(torch.bfloat16)
        w = (torch.randn(2 * I, Kd, device=dev, generator=gen) / Kd ** 0.5).to(torch.bfloat16)
        y = torch.empty(M, I, device=dev, dtype=torch.bfloat16)
        h = torch.empty(M, 2 * I, device=dev, dtype=torch.bfloat16)
        wg, wu = w[:I], w[I:]

        def fused():
            st = L.glu_gemm_fwd(x.data_ptr(), Kd, wg.data_ptr(), wu.data_ptr(), Kd, y.data_ptr(), I, M, Kd, I, 0,
                                2, s)
            if st:
                raise glu.GluError(st, "glu_gemm_fwd")

        def unfused():
            torch.matmul(x, w.T, out=h)
            st = L.glu_fwd(h.data_ptr(), 2 * I, None, 0, y.data_ptr(), I, M, I, 1, 0, 2, s)
            if st:
                raise glu.GluError(st, "glu_fwd")

        f_ms = timed(fused, K, W)
        info = glu.glu_last_launch()
        g_ms = timed(lambda: torch.matmul(x, w.T, out=h), K, W)
        u_ms = timed(unfused, K, W)
        fl = 2 * M * Kd * 2 * I
        out.append({"M": M, "K": Kd, "I": I, "fused_ms": round(f_ms, 4),
                    "fused_tflops": round(fl / (f_ms * 1e-3) / 1e12, 1),
                    "weights_gbs": round(2 * I * Kd * 2 / (f_ms * 1e-3) / 1e9, 1),
                    "cublas_gemm_ms": round(g_ms, 4), "cublas_gemm_plus_glu_fwd_ms": round(u_ms, 4),
                    "vs_cublas_gemm": round(g_ms / f_ms, 3), "vs_unfused": round(u_ms / f_ms, 3),
                    "tile_columns": tile_columns(M, I, info), "tiles": info["vector_units"],
                    "cluster": info["unroll"]})
        del x, w, y, h
    return out


def run_gemm(args):
    """The gate/up projections with SwiGLU in the epilogue (glu_gemm_fwd) on one
    MLP layer, against the unfused path it replaces: one cuBLAS GEMM into a
    [gate | up] matrix, then glu_fwd over it.  Operands (x 32 MiB, weights
    224 MiB) exceed L2.  Prints one JSON line (not the headline metric)."""
    import torch
    import glu_activation_mlps_gb300 as glu

    glu.build()
    L = glu.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    gen = torch.Generator(device=dev).manual_seed(7)
    x = torch.randn(GM, GK, device=dev, generator=gen).to(torch.bfloat16)
    w = (torch.randn(2 * GI, GK, device=dev, generator=gen) / GK ** 0.5).to(torch.bfloat16)
    wg, wu = w[:GI], w[GI:]
    y = torch.empty(GM, GI, device=dev, dtype=torch.bfloat16)
    h = torch.empty(GM, 2 * GI, device=dev, dtype=torch.bfloat16)
    stream = torch.cuda.current_stream()
    s = stream.cuda_stream
    flops = 2 * GM * GK * 2 * GI

    def fused():
        st = L.glu_gemm_fwd(x.data_ptr(), GK, wg.data_ptr(), wu.data_ptr(), GK, y.data_ptr(), GI,
                            GM, GK, GI, 0, 2, s)
        if st:
            raise glu.GluError(st, "glu_gemm_fwd")

    def unfused():
        torch.matmul(x, w.T, out=h)
        st = L.glu_fwd(h.data_ptr(), 2 * GI, None, 0, y.data_ptr(), GI, GM, GI, 1, 0, 2, s)
        if st:
            raise glu.GluError(st, "glu_fwd")

    def timed(fn, K, W, clocks=None):
        for _ in range(W):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        if clocks:
            clocks.mark(True)
        e0.record(stream)
        for _ in range(K):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        if clocks:
            clocks.mark(False)
        return e0.elapsed_time(e1) / K

    K, W = max(1, args.steps), max(3, args.warmup)
    clocks = ClockSampler(gpu_selector(0))
    clocks.start()
    fused_ms = timed(fused, K, W, clocks)
    clock_info = clocks.stop()
    info = glu.glu_last_launch()
    # the same clock record for cuBLAS's GEMM: under the power cap the two
    # kernels can run at different SM clocks, which the ratio of times includes
    gemm_clocks = ClockSampler(gpu_selector(0))
    gemm_clocks.start()
    gemm_ms = timed(lambda: torch.matmul(x, w.T, out=h), K, W, gemm_clocks)
    gemm_clock_info = gemm_clocks.stop()
    unfused_ms = timed(unfused, K, W)
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    peak = float(peaks["bf16_tflops"])
    tf = flops / (fused_ms * 1e-3) / 1e12
    shapes = gemm_shapes(L, glu, timed, dev, s, max(5, min(K, 50)), W) if not args.no_sweep else []
    line = {
        "metric": "gate/up projections with SwiGLU in the epilogue, TFLOP/s (bf16, M=4096 K=4096 I=14336)",
        "value": round(tf, 1), "unit": "TFLOP/s", "n_gpus": 1, "steps": K, "warmup": W,
        "ms_per_step": round(fused_ms, 5), "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "one MLP layer's gate/up projections: x 4096x4096, w_gate and w_up "
                               "14336x4096 (N(0,1) and N(0,1/4096), bf16), y 4096x14336",
                   "l2": "operands (256 MiB) exceed L2", "launch": info},
        "roofline": {"bound": "tensor", "kernel": "glu_gemm_fwd", "achieved": round(tf, 1), "peak": peak,
                     "peak_source": "measured (MEASURED_PEAKS.json bf16_tflops, cuBLAS burst)",
                     "unit": "TFLOP/s", "frac": round(tf / peak, 4), "traffic": None,
                     "algorithmic_flops": flops},
        "comparison": {"fused_ms": round(fused_ms, 4),
                       "cublas_gemm_ms": round(gemm_ms, 4),
                       "cublas_gemm_tflops": round(flops / (gemm_ms * 1e-3) / 1e12, 1),
                       "cublas_gemm_plus_glu_fwd_ms": round(unfused_ms, 4),
                       "speedup_vs_unfused": round(unfused_ms / fused_ms, 4),
                       "cublas_gemm_clocks": gemm_clock_info},
        "shapes": shapes,
        "gpu_launches": K,
        "clocks": clock_info,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- the whole gated MLP

def run_mlp(args):
    """glu_mlp_fwd on one decoder layer's MLP (4096 tokens, hidden 4096,
    intermediate 14336, bf16, SwiGLU): the gate/up GEMM with the activation in
    its epilogue, then the down GEMM, in row chunks whose y stays in L2.
    Against the unfused path (cuBLAS GEMM into [gate | up], glu_fwd, cuBLAS
    down GEMM) and against glu_gemm_fwd + glu_gemm_nt over all rows at once (y
    through HBM), all in one process.  Prints one JSON line."""
    import torch
    import glu_activation_mlps_gb300 as glu

    glu.build()
    L = glu.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    gen = torch.Generator(device=dev).manual_seed(9)
    M, H, I = GM, GK, GI
    x = torch.randn(M, H, device=dev, generator=gen).to(torch.bfloat16)
    w = (torch.randn(2 * I, H, device=dev, generator=gen) / H ** 0.5).to(torch.bfloat16)
    wg, wu = w[:I], w[I:]
    wd = (torch.randn(H, I, device=dev, generator=gen) / I ** 0.5).to(torch.bfloat16)
    out = torch.empty(M, H, device=dev, dtype=torch.bfloat16)
    y = torch.empty(M, I, device=dev, dtype=torch.bfloat16)
    h = torch.empty(M, 2 * I, device=dev, dtype=torch.bfloat16)
    ws_bytes = L.glu_mlp_workspace_bytes(M, I, 2)
    ws = torch.empty(ws_bytes, device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream()
    s = stream.cuda_stream
    flops = 2 * M * H * 2 * I + 2 * M * I * H

    def fused():
        st = L.glu_mlp_fwd(x.data_ptr(), H, wg.data_ptr(), wu.data_ptr(), H, wd.data_ptr(), I, out.data_ptr(), H,
                           M, H, I, 0, 2, ws.data_ptr(), ws_bytes, s)
        if st:
            raise glu.GluError(st, "glu_mlp_fwd")

    def whole():
        st = L.glu_gemm_fwd(x.data_ptr(), H, wg.data_ptr(), wu.data_ptr(), H, y.data_ptr(), I, M, H, I, 0, 2, s)
        if st:
            raise glu.GluError(st, "glu_gemm_fwd")
        st = L.glu_gemm_nt(y.data_ptr(), I, wd.data_ptr(), I, out.data_ptr(), H, M, I, H, 2, s)
        if st:
            raise glu.GluError(st, "glu_gemm_nt")

    def unfused():
        torch.matmul(x, w.T, out=h)
        st = L.glu_fwd(h.data_ptr(), 2 * I, None, 0, y.data_ptr(), I, M, I, 1, 0, 2, s)
        if st:
            raise glu.GluError(st, "glu_fwd")
        torch.matmul(y, wd.T, out=out)

    def timed(fn, K, W, clocks=None):
        for _ in range(W):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        if clocks:
            clocks.mark(True)
        e0.record(stream)
        for _ in range(K):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        if clocks:
            clocks.mark(False)
        return e0.elapsed_time(e1) / K

    K, W = max(1, args.steps), max(3, args.warmup)
    clocks = ClockSampler(gpu_selector(0))
    clocks.start()
    fused_ms = timed(fused, K, W, clocks)
    clock_info = clocks.stop()
    whole_ms = timed(whole, K, W)
    unfused_ms = timed(unfused, K, W)
    down_ms = timed(lambda: torch.matmul(y, wd.T, out=out), K, W)
    nt_ms = timed(lambda: L.glu_gemm_nt(y.data_ptr(), I, wd.data_ptr(), I, out.data_ptr(), H, M, I, H, 2, s), K, W)
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    peak = float(peaks["bf16_tflops"])
    tf = flops / (fused_ms * 1e-3) / 1e12
    down_flops = 2 * M * I * H
    line = {
        "metric": "gated MLP (gate/up GEMM + SwiGLU + down GEMM), TFLOP/s (bf16, M=4096 H=4096 I=14336)",
        "value": round(tf, 1), "unit": "TFLOP/s", "n_gpus": 1, "steps": K, "warmup": W,
        "ms_per_step": round(fused_ms, 5), "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "one decoder layer's MLP: x 4096x4096, w_gate and w_up 14336x4096, w_down "
                               "4096x14336 (N(0,1), N(0,1/4096), N(0,1/14336), bf16)",
                   "chunk_rows": ws_bytes // (2 * ((I + 7) // 8 * 8)), "workspace_bytes": ws_bytes},
        "roofline": {"bound": "tensor", "kernel": "glu_mlp_fwd", "achieved": round(tf, 1), "peak": peak,
                     "peak_source": "measured (MEASURED_PEAKS.json bf16_tflops, cuBLAS burst)",
                     "unit": "TFLOP/s", "frac": round(tf / peak, 4), "traffic": None, "algorithmic_flops": flops},
        "comparison": {"fused_ms": round(fused_ms, 4),
                       "glu_gemm_fwd_then_glu_gemm_nt_all_rows_ms": round(whole_ms, 4),
                       "cublas_gemm_glu_fwd_cublas_gemm_ms": round(unfused_ms, 4),
                       "speedup_vs_unfused": round(unfused_ms / fused_ms, 4),
                       "glu_gemm_nt_down_ms": round(nt_ms, 4), "cublas_down_ms": round(down_ms, 4),
                       "glu_gemm_nt_vs_cublas": round(down_ms / nt_ms, 4),
                       "glu_gemm_nt_tflops": round(down_flops / (nt_ms * 1e-3) / 1e12, 1)},
        "gpu_launches": K * 2 * -(-M // (ws_bytes // (2 * ((I + 7) // 8 * 8)))),
        "clocks": clock_info,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- residual add + RMSNorm

def run_rmsnorm(args):
    """glu_add_rmsnorm_fwd on one decoder block's residual add + RMSNorm (4096
    tokens x hidden 4096, bf16, eps 1e-5, rstd kept), and an H sweep, against
    torch's unfused path (an add kernel, then F.rms_norm).  Each timed launch
    uses the next of several buffer sets whose total exceeds L2.  Prints one
    JSON line (not the headline metric)."""
    import torch
    import torch.nn.functional as F
    import glu_activation_mlps_gb300 as glu

    glu.build()
    L = glu.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    s = stream.cuda_stream
    gen = torch.Generator(device=dev).manual_seed(8)
    peak, peak_src = measured_peak()
    K, W = max(1, args.steps), max(3, args.warmup)

    def timed(fn, nsets, clocks=None):
        for k in range(W):
            fn(k % nsets)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        if clocks:
            clocks.mark(True)
        e0.record(stream)
        for k in range(K):
            fn(k % nsets)
        e1.record(stream)
        torch.cuda.synchronize()
        if clocks:
            clocks.mark(False)
        return e0.elapsed_time(e1) / K

    def case(rows, H, clocks=None):
        E = 2
        per_set = 4 * rows * H * E
        nsets = max(2, -(-3 * L2_BYTES // per_set))
        sets = []
        for _ in range(nsets):
            x = torch.randn(rows, H, device=dev, generator=gen).to(torch.bfloat16)
            r = (torch.randn(rows, H, device=dev, generator=gen) * 4).to(torch.bfloat16)
            sets.append((x, r, torch.empty_like(x), torch.empty_like(x)))
        g = (1 + 0.1 * torch.randn(H, device=dev, generator=gen)).to(torch.bfloat16)
        rstd = torch.empty(rows, device=dev, dtype=torch.float32)

        def fused(k):
            x, r, h, y = sets[k]
            st = L.glu_add_rmsnorm_fwd(x.data_ptr(), H, r.data_ptr(), H, g.data_ptr(), h.data_ptr(), H,
                                       y.data_ptr(), H, rstd.data_ptr(), rows, H, 1e-5, 2, s)
            if st:
                raise glu.GluError(st, "glu_add_rmsnorm_fwd")

        def unfused(k):
            x, r, h, y = sets[k]
            torch.add(x, r, out=h)
            y.copy_(F.rms_norm(h, (H,), g, 1e-5))

        ms = timed(fused, nsets, clocks)
        info = glu.glu_last_launch()
        ms_unfused = timed(unfused, nsets)
        nbytes = 4 * rows * H * E + H * E + 4 * rows
        return {"rows": rows, "H": H, "ms": round(ms, 5), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                "frac": round(nbytes / (ms * 1e-3) / 1e9 / peak, 4), "torch_unfused_ms": round(ms_unfused, 5),
                "speedup_vs_unfused": round(ms_unfused / ms, 3), "bytes": nbytes, "launch": info,
                "buffer_sets": nsets}

    def backward(rows, H):
        """glu_add_rmsnorm_bwd (dx, dgamma) against torch autograd through add +
        F.rms_norm; algorithmic bytes: read dy and h, write dx (3 row passes)."""
        E = 2
        nsets = max(2, -(-3 * L2_BYTES // (3 * rows * H * E)))
        sets = [((torch.randn(rows, H, device=dev, generator=gen)).to(torch.bfloat16),
                 (torch.randn(rows, H, device=dev, generator=gen) * 4).to(torch.bfloat16),
                 torch.empty(rows, H, device=dev, dtype=torch.bfloat16)) for _ in range(nsets)]
        g = (1 + 0.1 * torch.randn(H, device=dev, generator=gen)).to(torch.bfloat16)
        rstd = (0.2 + 0.5 * torch.rand(rows, device=dev, generator=gen)).float()
        dgam = torch.zeros(H, device=dev, dtype=torch.float32)

        def fused(k):
            dy, h, dx = sets[k]
            st = L.glu_add_rmsnorm_bwd(dy.data_ptr(), H, h.data_ptr(), H, rstd.data_ptr(), g.data_ptr(), None, 0,
                                       dx.data_ptr(), H, None, 0, dgam.data_ptr(), rows, H, 2, s)
            if st:
                raise glu.GluError(st, "glu_add_rmsnorm_bwd")

        ms = timed(fused, nsets)
        info = glu.glu_last_launch()
        # torch: the same gradients through autograd of add + rms_norm
        xs = [sets[k][1].clone().requires_grad_(True) for k in range(nsets)]
        gt = g.clone().requires_grad_(True)
        graphs = [F.rms_norm(xs[k] + 0, (H,), gt, 1e-5) for k in range(nsets)]

        def unfused(k):
            torch.autograd.grad(graphs[k], (xs[k], gt), sets[k][0], retain_graph=True)

        ms_t = timed(unfused, nsets)
        nbytes = 3 * rows * H * E + H * E + 4 * rows + 4 * H
        return {"rows": rows, "H": H, "ms": round(ms, 5), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                "frac": round(nbytes / (ms * 1e-3) / 1e9 / peak, 4), "torch_autograd_ms": round(ms_t, 5),
                "speedup_vs_torch": round(ms_t / ms, 3), "bytes": nbytes, "launch": info}

    clocks = ClockSampler(gpu_selector(0))
    clocks.start()
    main = case(4096, 4096, clocks)
    clock_info = clocks.stop()
    sweep = [case(4096, H) for H in (1024, 2048, 8192, 16384)]
    bwd = [backward(4096, H) for H in (512, 1024, 2048, 4096, 8192, 16384)]
    line = {
        "metric": "fused residual add + RMSNorm achieved HBM GB/s (bf16, 4096 tokens x hidden 4096)",
        "value": main["gbs"], "unit": "GB/s", "n_gpus": 1, "steps": K, "warmup": W,
        "ms_per_step": main["ms"], "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "h = x + residual, y = rmsnorm(h) * gamma, eps 1e-5, rstd kept; x ~ N(0,1), "
                               "residual ~ N(0,4^2), gamma ~ 1 + N(0,0.1^2)",
                   "l2": f"each launch uses the next of {main['buffer_sets']} buffer sets (together > L2)",
                   "launch": main["launch"]},
        "roofline": {"bound": "hbm", "kernel": "glu_add_rmsnorm_fwd", "achieved": main["gbs"], "peak": peak,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, copy)", "unit": "GB/s",
                     "frac": main["frac"], "traffic": None, "algorithmic_bytes": main["bytes"]},
        "comparison": {"torch_add_then_rms_norm_ms": main["torch_unfused_ms"],
                       "speedup_vs_unfused": main["speedup_vs_unfused"]},
        "sweep": [{k: c[k] for k in ("rows", "H", "ms", "gbs", "frac", "torch_unfused_ms", "speedup_vs_unfused")}
                  for c in sweep],
        "backward": bwd,
        "gpu_launches": K,
        "clocks": clock_info,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- CPU oracle arms

def oracle_rows(orc, d, r0, r1, threads):
    a, b, dc = d["a"][r0:r1], d["b"][r0:r1], d["dc"][r0:r1]
    orc.fwd_threaded("silu", "bf16", a, b, threads)
    orc.bwd_threaded("silu", "bf16", dc, a, b, threads)


def oracle_gbs(orc, d, threads, budget_s):
    """The oracle's throughput (forward + backward, algorithmic bytes over
    wall time) on `threads` host threads.  One untimed call first (thread
    start-up, first touch of the outputs, clock ramp), then a call on 16 rows
    sizes the blocks so that one call takes about a quarter of `budget_s`;
    blocks of consecutive rows are timed until `budget_s` has passed.
    Returns (GB/s, rows timed, seconds timed, rows per call)."""
    oracle_rows(orc, d, 0, 16, threads)
    t = time.perf_counter()
    oracle_rows(orc, d, 0, 16, threads)
    per_row = (time.perf_counter() - t) / 16
    block = int(max(16, min(ROWS, budget_s / 4 / max(per_row, 1e-9))))
    spent, done, r0 = 0.0, 0, 0
    while spent < budget_s:
        if r0 + block > ROWS:
            r0 = 0
        s = time.perf_counter()
        oracle_rows(orc, d, r0, r0 + block, threads)
        spent += time.perf_counter() - s
        done += block
        r0 += block
    return done * COLS * 8 * E / spent / 1e9, done, spent, block


def cpu_baseline(d, budget_s=3.0):
    """The oracle, as it stands, on the host cores: all of them (the reported
    value) and one, each timed for about `budget_s` seconds after a warm-up
    call (oracle_gbs)."""
    import oracle as orc
    orc.build()
    threads = os.cpu_count() or 1
    gbs, rows, secs, block = oracle_gbs(orc, d, threads, budget_s)
    gbs1, rows1, secs1, block1 = oracle_gbs(orc, d, 1, budget_s)

    def sample(r, sec, blk, th):
        return (f"{r} rows of the 4096x14336 bf16 workload in blocks of {blk} rows (fwd + bwd, "
                f"{r * COLS} elements, {sec:.2f} s on {th} thread{'s' if th > 1 else ''}, after one "
                f"untimed call)")
    return {"value": round(gbs, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": sample(rows, secs, block, threads),
            "all_cores": {"value": round(gbs, 3), "cores": threads},
            "single_thread": {"value": round(gbs1, 3), "cores": 1, "sample": sample(rows1, secs1, block1, 1)}}


def run_reference(args):
    """The double-precision CPU oracle timed as the reference arm: every step
    runs forward + backward on a block of rows of the same workload."""
    import oracle as orc
    orc.build()
    d = glu_synth.metric_bf16()
    threads = os.cpu_count() or 1
    t0 = time.perf_counter()
    oracle_rows(orc, d, 0, 16, threads)
    per_row = (time.perf_counter() - t0) / 16
    total_steps = args.steps + args.warmup
    rows = int(max(1, min(ROWS, args.ref_seconds / max(total_steps, 1) / max(per_row, 1e-9))))
    for k in range(args.warmup):
        oracle_rows(orc, d, 0, rows, threads)
    times = []
    for k in range(args.steps):
        s = time.perf_counter()
        oracle_rows(orc, d, 0, rows, threads)
        times.append(time.perf_counter() - s)
    total = sum(times)
    nbytes = rows * COLS * 8 * E
    value = args.steps * nbytes / total / 1e9
    sample = f"rows 0..{rows} of the 4096x14336 bf16 workload per step (fwd + bwd, {rows * COLS} elements)"
    # beside it, the same oracle on one thread (a short bounded sample)
    gbs1, rows1, secs1, block1 = oracle_gbs(orc, d, 1, min(10.0, args.ref_seconds / 6))
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config({"parallelism": f"{threads} host threads", "math": "f64"}),
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample, "all_cores": {"value": round(value, 3), "cores": threads},
                         "single_thread": {"value": round(gbs1, 3), "cores": 1,
                                           "sample": f"{rows1} rows in blocks of {block1} rows, {secs1:.2f} s "
                                                     "on 1 thread, after one untimed call"}},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=3.0)
    ap.add_argument("--ref-seconds", type=float, default=90.0)
    ap.add_argument("--gemm", action="store_true",
                    help="time glu_gemm_fwd on one MLP layer against cuBLAS + glu_fwd (one JSON line)")
    ap.add_argument("--no-sweep", action="store_true",
                    help="--gemm: skip the other layer shapes")
    ap.add_argument("--mlp", action="store_true",
                    help="time glu_mlp_fwd on one decoder layer's MLP against cuBLAS + glu_fwd + cuBLAS")
    ap.add_argument("--rmsnorm", action="store_true",
                    help="time glu_add_rmsnorm_fwd on one decoder block against torch's add + rms_norm")
    ap.add_argument("--table", action="store_true",
                    help="print a throughput table of every named workload instead of the JSON line")
    ap.add_argument("--path", default="default", choices=["default", "direct", "bulk"],
                    help="load path of the kernels (library default, direct loads, or bulk copies "
                         "staged in shared memory); for profiling and comparisons")
    ap.add_argument("--case", default=None,
                    help="launch one named workload (" + ", ".join(CASES) + ", or sweep:<act>:<dtype>:<dir>:<H>) "
                         "--warmup + --steps times and print its per-launch time (the command the per-config "
                         "ncu captures profile)")
    ap.add_argument("--graph", type=int, default=0,
                    help="--case: capture N repetitions of the case into one CUDA graph and time its replays")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.case:
        run_case(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.gemm:
        run_gemm(args)
        return
    if args.mlp:
        run_mlp(args)
        return
    if args.rmsnorm:
        run_rmsnorm(args)
        return
    if args.table:
        run_table(args)
        return

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        line = run_gpu(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
