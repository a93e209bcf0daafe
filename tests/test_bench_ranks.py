"""The multi-rank bookkeeping of bench.py on CPU: world size 2 over gloo, every
rank receives the slowest rank's time, and the whole-job value counts every
replica's bytes against that time."""
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


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
        got = bench.max_over_ranks(ms, dist, device="cpu")
        value = bench.replica_value(world, 1e9, 4, got)
        out.put((rank, got, value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_replica_value_gloo_world_2():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, got, value in res:
        assert got == 15.0
        assert value == pytest.approx(2 * 1e9 * 4 / 15e-3 / 1e9)


def test_single_rank_passthrough():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.replica_value(1, 2e9, 10, 20.0) == pytest.approx(1000.0)
