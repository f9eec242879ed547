"""The multi-process (N > 1) paths of bench.py on CPU, with the gloo backend.

One GEMM needs no collective ("replicas only": every rank runs its own
problem), so the only cross-rank steps are the barriers around the timed
region and the maximum of the ranks' elapsed times.  Both are checked here
with world_size 2 on gloo; the reference arm is also run under torchrun
exactly as the driver launches it, with rank 0 alone printing its line.
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


def _max_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(dist)
        # rank r "measured" 10 * (r + 1) ms: every rank must report the slowest
        got = bench.max_over_ranks(dist, 10.0 * (rank + 1), torch.device("cpu"))
        out[rank] = got
        bench.barrier(dist)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_max_worker, args=(world, free_port(), out), nprocs=world, join=True)
    assert dict(out) == {0: 20.0, 1: 20.0}


def test_single_rank_max_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 3.25, None) == 3.25


@pytest.mark.timeout(600)
def test_reference_arm_under_torchrun_two_ranks():
    """The driver's launch line with --nproc-per-node 2: rank 0 prints one JSON
    line for the reference arm, rank 1 exits 0 without work."""
    from oracle import build
    build()
    env = dict(os.environ, OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "gemm512_uniform", "--gpus", "2", "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["unit"] == "TFLOP/s"
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
