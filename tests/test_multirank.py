"""Host-side logic of the N > 1 bench path on CPU with gloo, world size 2.

Each rank runs the whole workload on its own device (independent batches, weak
scaling); the only collectives are the timing barrier and the max/sum of the
ranks' scalars.  Nothing here needs a GPU.
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


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    bench.init_dist(world, "gloo")
    try:
        w, r, _ = bench.dist_env()
        bench.barrier(w)
        slowest = bench.max_over_ranks(10.0 + r, w)           # rank 1 is the slow one
        total = bench.sum_over_ranks(100.0 * (r + 1), w)
        seeds = [bench.rank_seed_offset(k) for k in range(w)]
        q.put((r, w, slowest, total, seeds))
    finally:
        dist.destroy_process_group()


def test_two_rank_reductions():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(world))
    for r, w, slowest, total, seeds in res:
        assert w == 2
        assert slowest == 11.0          # max over ranks
        assert total == 300.0           # sum over ranks
        assert len(set(seeds)) == 2     # each rank draws its own batch


def test_reference_arm_under_torchrun_rank1_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0", "--gpus", "2"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_reference_arm_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "1"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
