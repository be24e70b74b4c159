"""Replicas-only multi-GPU path, host side, on CPU: two gloo ranks.

Requests are independent and the drafter keeps no state across rounds, so N
GPUs run N replicas with no data-path collective; the bench's only exchange is
the timing reduction (the slowest rank's seconds, the sum of committed tokens)
and each rank drafts its own shard of requests.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from history_free_speculative_gb300 import workload as wk
        ws, r, local = bench.dist_env()
        t_s, committed = bench.reduce_over_ranks(0.5 + rank, 10 * (rank + 1), "cpu")
        wl = wk.WORKLOADS["tiny"]
        hidden, _, _ = wk.make_round_inputs(wl, round_index=bench.shard_round_index(0, rank))
        out.put((rank, ws, r, t_s, committed, float(hidden.double().sum())))
    finally:
        dist.destroy_process_group()


def test_two_replicas_reduce_time_and_tokens():
    ctx = mp.get_context("spawn")
    out = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(out.get() for _ in range(2))
    for rank, ws, r, t_s, committed, _ in res:
        assert (ws, r) == (2, rank)
        assert t_s == 1.5           # the slowest rank's time
        assert committed == 30      # every rank's committed tokens
    assert res[0][5] != res[1][5]   # each replica drafts its own requests


def test_single_process_reduction_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(0.25, 7, "cpu") == (0.25, 7)
    assert bench.shard_round_index(3, 0) == 3 and bench.shard_round_index(3, 1) != 3


def test_bench_rejects_gpus_that_disagree_with_the_launcher():
    """Under a launcher the rank count is WORLD_SIZE; a --gpus that disagrees is an error
    (without a launcher, --gpus N > 1 starts N ranks itself)."""
    import subprocess
    import sys
    env = dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "4", "--steps", "1"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0 and "WORLD_SIZE is 2" in r.stderr
