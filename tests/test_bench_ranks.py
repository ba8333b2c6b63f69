"""The benchmark's multi-rank arithmetic on two gloo ranks (CPU only).

With torchrun every rank runs its own replica of the workload (weak scaling,
no data-path collective); the step time is the maximum over ranks and the
reported throughput counts the units of all ranks.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, units, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    slowest = bench.max_over_ranks(times[rank], dist, world)
    rate = bench.whole_job_rate(units, world, slowest)
    out[rank] = (slowest, rate)
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_step_and_count_all_units():
    world, port = 2, _free_port()
    times = [0.125, 0.5]
    units = 4096
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, times, units, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        slowest, rate = res[r]
        assert slowest == pytest.approx(0.5)
        assert rate == pytest.approx(units * world / 0.5)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(0.25, None, 1) == 0.25
    assert bench.whole_job_rate(100, 1, 0.5) == 200
