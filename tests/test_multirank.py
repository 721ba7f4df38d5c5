"""The multi-process (N > 1) host logic of bench.py, on CPU with gloo, world size 2.

The path shards into independent (b, h) heads / query blocks, so ranks run
independent replicas; the only cross-rank operations are the timing barrier and
the max-over-ranks reduction, which these tests exercise.
"""
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


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    d, r, w, local = bench.dist_setup(world)
    assert d is not None and r == rank and w == world
    bench.barrier(d)
    mx = bench.max_over_ranks(d, float(rank + 1) * 10.0)
    sm = bench.sum_over_ranks(d, float(rank + 1))
    results[rank] = (mx, sm)
    dist.destroy_process_group()


def test_gloo_barrier_and_max_over_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_worker, args=(world, free_port(), results), nprocs=world,
                           start_method="spawn", join=True)
        assert dict(results) == {0: (20.0, 3.0), 1: (20.0, 3.0)}


def test_reference_arm_under_torchrun_prints_one_line_from_rank0():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--workload", "tiny", "--steps", "1", "--warmup", "3", "--ref-step-s", "0.2"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["e2e"]["h2d_bytes_per_step"] == 0
