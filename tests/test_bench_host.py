"""Host-side logic of bench.py on the CPU: the max-over-ranks reduction and
the whole-job throughput with two gloo ranks, and the reference arm (the
oracle on the host cores) launched the way the driver launches N > 1 runs,
where rank 0 alone prints one JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        my_ms = 10.0 + 5.0 * rank                  # rank 1 is the slowest
        ms = bench.reduce_max(my_ms)
        out[rank] = (ms, bench.job_gbs(world, 100, bench.STEP_BYTES, ms))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_with_gloo():
    world, port = 2, free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]                        # every rank agrees
    ms, gbs = res[0]
    assert ms == 15.0                              # the slowest rank's time
    assert gbs == pytest.approx(2 * 100 * bench.STEP_BYTES / 0.015 / 1e9)


def test_reduce_max_without_process_group_is_identity():
    assert bench.reduce_max(3.25) == 3.25
    assert bench.job_gbs(1, 10, 1_000_000_000, 1000.0) == pytest.approx(10.0)


def test_reference_arm_under_torchrun_prints_one_line(tmp_path):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "3", "--warmup", "3", "--ref-seconds", "2"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["metric"] == bench.METRIC


def test_warmup_below_three_is_rejected():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode != 0 and "warmup" in r.stderr
