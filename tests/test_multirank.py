"""Replica (weak-scaling) aggregation of bench.py across ranks, on CPU with
gloo at world size 2: the slowest rank's time sets the step time, and the
job's value counts every rank's bytes."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = [1.0 + rank, 10.0 - rank, 5.0]
    got = bench.max_over_ranks(mine, torch.device("cpu"), world)
    dist.barrier()
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q))
             for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [2.0, 10.0, 5.0]


def test_aggregate_value_counts_all_ranks():
    import bench
    one = bench.aggregate_value(6e8, 0.1, 1)
    assert bench.aggregate_value(6e8, 0.1, 4) == pytest.approx(4 * one)
    assert one == pytest.approx(6000.0)
