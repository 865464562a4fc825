"""The multi-rank path of bench.py, on CPU with two gloo ranks.

The norm and the compose shard with no exchange (every module and every row
is independent), so N GPUs run N independent modules: rank k draws its own
inputs (seed k), and the only collectives are the timing contract's barrier
and the maximum of the per-rank times.  The reference arm runs on rank 0
alone; the other ranks exit at once without output."""
from __future__ import annotations

import argparse
import hashlib
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q) -> None:
    sys.path.insert(0, ROOT)
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        import bench
        from synthetic import configs, gen
        env = bench.dist_env()
        # per-rank times: the job's time is the slowest rank's
        slowest = bench.max_over_ranks(1.5 * (rank + 1), env[0], torch.device("cpu"))
        bench.barrier(env[0])
        x = gen.norm_inputs(configs.get(0), seed=rank)
        digests = [None] * world
        dist.all_gather_object(digests, hashlib.sha256(x["W"].tobytes()).hexdigest())
        ref = None
        if rank != 0:
            ref = bench.run_reference(argparse.Namespace(steps=1, warmup=3))
        q.put((rank, env, slowest, digests, ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replica_path():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    world = 2
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = {}
    try:
        for _ in range(world):
            rank, env, slowest, digests, ref = q.get(timeout=180)
            results[rank] = (env, slowest, digests, ref)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert sorted(results) == [0, 1]
    for rank, (env, slowest, digests, ref) in results.items():
        assert env == (world, rank, rank)
        assert slowest == pytest.approx(3.0)          # max of 1.5 and 3.0 on both ranks
        assert digests[0] != digests[1]               # independent inputs per rank
        if rank != 0:
            assert ref == 0                           # reference arm: rank 0 only
    assert all(p.exitcode == 0 for p in procs)
