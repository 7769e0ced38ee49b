"""The multi-rank part of bench.py on CPU: two gloo ranks on 127.0.0.1 agree
on the slowest rank's time, and the whole-job rate counts every replica."""
import os
import socket

import pytest

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, results):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r "took" 10 * (r + 1) ms
        mx = bench.max_over_ranks(10.0 * (rank + 1), dist, "cpu")
        dist.barrier()
        results[rank] = mx
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    import torch.multiprocessing as mp
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
        assert dict(results) == {0: 20.0, 1: 20.0}


def test_whole_job_rate_counts_every_replica():
    flops = 2.0 * 8192 ** 3
    one = bench.whole_job_rate(1, flops, 100, 70.0)
    assert one == pytest.approx(flops * 100 / 0.070 / 1e12)
    assert bench.whole_job_rate(4, flops, 100, 70.0) == pytest.approx(4 * one)
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
