"""The multi-GPU path is independent replicas (one full evaluation per rank,
no collective on the data path). Its host-side aggregation -- max time over
ranks, units summed over ranks -- is checked here with two gloo ranks on CPU."""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    # rank r took (r + 1) * 10 ms over 5 steps and processed 1000 * (r + 1) units
    ms, value = bench.replica_throughput((rank + 1) * 10.0, 1000.0 * (rank + 1), 5, dist,
                                         torch.device("cpu"))
    q.put((rank, ms, value))
    dist.barrier()
    dist.destroy_process_group()


def test_replica_throughput_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, value in got:
        assert ms == pytest.approx(20.0 / 5)                       # slowest rank
        assert value == pytest.approx(3000.0 / (20.0 / 5 / 1000))  # all ranks' units


def test_replica_throughput_single_process():
    import bench

    ms, value = bench.replica_throughput(10.0, 500.0, 5)
    assert ms == pytest.approx(2.0) and value == pytest.approx(250000.0)
