"""The N > 1 path of bench.py on CPU: two gloo ranks (the replica aggregation
the GPU run does over NCCL) -- every rank gets the slowest rank's time and the
job throughput counts every replica's units."""
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


def _rank_main(rank, world, port, times, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], dist, torch.device("cpu"))
        dist.barrier()
        q.put((rank, ms, bench.job_throughput(2.0, world, ms)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, times = 2, [0.030, 0.045]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, ms, thr in got:
        assert ms == pytest.approx(0.045)
        assert thr == pytest.approx(2.0 * 2 / 0.045e-3)


def test_single_rank_helpers():
    import bench
    assert bench.max_over_ranks(0.5, None, None) == 0.5
    assert bench.job_throughput(3.0, 1, 1.0) == pytest.approx(3000.0)
