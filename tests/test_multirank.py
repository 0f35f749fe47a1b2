"""The N > 1 path on CPU with gloo, world size 2: bench.py runs one independent replica per rank
(weak scaling), reduces the timing to the slowest rank and prints from rank 0 only; the
reference arm runs on rank 0 alone."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(10.0 + 5.0 * rank, torch.device("cpu"), world)  # rank 1 is the slow one
        out[rank] = t
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1] == 15.0


def test_whole_job_value_is_weak_scaling():
    import importlib
    sys.path.insert(0, ROOT)
    bench = importlib.import_module("bench")
    one = bench.whole_job_value(89_194_496, 1, 0.036)
    assert abs(bench.whole_job_value(89_194_496, 2, 0.036) - 2 * one) < 1e-9
    assert abs(one - 89_194_496 / 36e-6 / 1e9) < 1e-6


def test_reference_arm_torchrun_world2():
    """`bench.py --impl reference` under torchrun with two CPU ranks: both exit 0, one JSON line."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "c1", "--gpus", "2", "--steps", "1", "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["n_gpus"] == 2 and res["value"] > 0
