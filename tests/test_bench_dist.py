"""bench.py's multi-rank plumbing on CPU: gloo at world size 2 (max-over-ranks
timing, barrier), and the reference arm under torchrun (rank 0 alone prints
one JSON line; the other rank exits 0 without work)."""

import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, lr = bench.dist_info()
    assert (r, w, lr) == (rank, world, rank)
    dist = bench.init_dist(world, "gloo")
    local_ms = 1.0 + rank  # rank 1 is the slow one
    ms = bench.max_over_ranks(local_ms, dist)
    bench.barrier(dist)
    with open(f"{path}.{rank}", "w") as fh:
        fh.write(repr(ms))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2(tmp_path):
    port = _free_port()
    mp.spawn(_worker, args=(2, port, str(tmp_path / "out")), nprocs=2, join=True)
    vals = [float(open(tmp_path / f"out.{r}").read()) for r in range(2)]
    assert vals == [2.0, 2.0]


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--ref-step-budget", "0.3", "--config", "config1"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_filter_workload_and_its_reference_arm():
    """The filter line's workload is config 2 with per-sequence top-k / top-p,
    and its reference arm runs the oracle with those filters."""
    import bench
    wl = bench.make_workload("filter")
    assert wl.B == 64 and wl.K == 5 and wl.V == 128256 and wl.dtype == "bf16"
    assert (wl.top_k == bench.FILTER_TOP_K).all() and np.allclose(wl.top_p, bench.FILTER_TOP_P)
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3",
           "--ref-step-budget", "0.3", "--config", "filter"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    d = json.loads([l for l in res.stdout.splitlines() if l.startswith("{")][-1])
    assert d["impl"] == "reference" and d["value"] > 0 and "top-k 50" in d["config"]["workload"]
