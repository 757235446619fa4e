"""The benchmark's replica aggregation over ranks, on CPU with gloo (world
size 2): each rank runs an independent replica of the codec (there is no
exchange step), and the job's figure is the total over ranks divided by the
slowest rank's time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        local_ms = 10.0 + 5.0 * rank  # rank 1 is slower
        dist.barrier()
        slowest = bench.max_over_ranks(local_ms, world, torch.device("cpu"))
        value = bench.replica_throughput_gbs(1 << 30, 4, slowest, world)
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_replica_aggregation_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, slowest, value in got:
        assert slowest == 15.0
        assert value == pytest.approx(2 * (1 << 30) * 4 / 0.015 / 1e9)


def test_single_rank_is_identity():
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.replica_throughput_gbs(1000, 2, 1.0, 1) == pytest.approx(2e-3)
