"""The N > 1 bench path is replicas (one frame per rank, no data-path
collective); its only cross-rank step is the max over ranks of the timings.
Checked here with two gloo ranks on CPU."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = [1.0 + rank, 5.0 - rank]          # rank 0 slower on the second value
    got = bench.max_over_ranks(mine)
    value, slowest = bench.aggregate([got[0]] * world, [1920 * 1080] * world)
    results[rank] = (got, value, slowest)
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_aggregate_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    procs = [ctx.Process(target=_rank, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(world):
        got, value, slowest = results[r]
        assert got == [2.0, 5.0]
        assert slowest == 2.0
        assert value == pytest.approx(2 * 1920 * 1080 / 1e6 / 2e-3)


def test_single_process_reduction_is_identity():
    import bench
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert bench.aggregate([2.0], [1000000])[0] == pytest.approx(500.0)
