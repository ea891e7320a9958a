"""The bench's multi-GPU mode runs one replica of the layer per rank (the
path has no exchange step): the job's time is the slowest rank's, and N
replicas finish N steps in it. Checked with two gloo ranks on the CPU."""
import os
import socket
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


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms_local = [10.0, 12.5][rank]          # rank 1 is the slower one
        q.put((rank, bench.replica_timing(ms_local, 100, world, "cpu")))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = dict(q.get(timeout=10) for _ in range(2))
    for r in range(2):
        job, rep = res[r]
        assert rep == pytest.approx(125.0)      # 12.5 ms over 100 steps, every rank
        assert job == pytest.approx(62.5)       # two replicas: two steps in that time


def test_single_rank_is_the_replica():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.replica_timing(5.0, 50, 1) == (100.0, 100.0)
