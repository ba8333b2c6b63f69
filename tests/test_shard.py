"""Sequence sharding across ranks (CPU only: gloo ranks, the fp64 oracle as each rank's compute).

Every (sequence, head) of the verification and of the commit is independent,
so a batch split by sequence over ranks, each rank verifying and committing
its own block, must gather to exactly the one-rank result -- bit for bit,
since each sequence's arithmetic is the same whichever rank runs it.  Also
checks the partition itself and the benchmark's launch logic for --gpus.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from speculative_decoding_linear_gb300 import shard
from speculative_decoding_linear_gb300 import workloads as wl


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("B,world", [(16, 2), (7, 2), (5, 3), (2, 4), (64, 8), (1, 1)])
def test_sequence_range_is_a_balanced_partition(B, world):
    blocks = [shard.sequence_range(B, world, r) for r in range(world)]
    assert blocks[0][0] == 0 and blocks[-1][1] == B
    for (lo0, hi0), (lo1, hi1) in zip(blocks, blocks[1:]):
        assert hi0 == lo1                                  # contiguous, no gap, no overlap
    sizes = [hi - lo for lo, hi in blocks]
    assert max(sizes) - min(sizes) <= 1 and sizes == sorted(sizes, reverse=True)
    assert sum(shard.gather_order(B, world), []) == list(range(B))


def test_sequence_range_rejects_bad_requests():
    for args in ((4, 0, 0), (4, 2, 2), (4, 2, -1), (-1, 2, 0)):
        with pytest.raises(ValueError):
            shard.sequence_range(*args)


def test_shard_keeps_weights_and_slices_sequences():
    w = wl.make_layer_workload(4, B=5, N=6, H=2, dk=16, dv=16, hidden=64)
    parts = [shard.shard_workload(w, 2, r) for r in range(2)]
    assert [p.B for p in parts] == [3, 2] and [p.spec.B for p in parts] == [3, 2]
    for name in ("X", "conv_state", "parent", "S0", "path"):
        assert np.array_equal(np.concatenate([getattr(p, name) for p in parts]), getattr(w, name))
    for name in ("W_in", "W_o", "conv_w"):
        assert all(getattr(p, name) is getattr(w, name) for p in parts)


def _oracle_block(w):
    x = dict(q=w.widened("q"), k=w.widened("k"), v=w.widened("v"), alpha=w.alpha.astype(np.float64),
             beta=w.beta.astype(np.float64), parent=w.parent, S0=w.S0.astype(np.float64))
    o, d, g = oracle.tree_verify(**x, nthreads=1)
    S = oracle.commit(x["k"], x["v"], x["alpha"], x["beta"], w.parent, x["S0"], w.path, nthreads=1)
    return o, d, g, S


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = wl.make_workload(wl.dataclasses.replace(wl.SPECS[3], B=5, H=2, dk=32, dv=16, N=12))
    mine = shard.shard_workload(w, world, rank)
    res = _oracle_block(mine)
    gathered = []
    for x in res:
        t = torch.from_numpy(np.ascontiguousarray(x))
        # blocks differ in size: pad to the largest, gather, cut back
        nmax = max(hi - lo for lo, hi in (shard.sequence_range(w.B, world, r) for r in range(world)))
        pad = torch.zeros((nmax,) + tuple(t.shape[1:]), dtype=t.dtype)
        pad[: t.shape[0]] = t
        bufs = [torch.zeros_like(pad) for _ in range(world)]
        dist.all_gather(bufs, pad)
        parts = [bufs[r][: hi - lo] for r, (lo, hi) in enumerate(shard.sequence_range(w.B, world, r)
                                                                   for r in range(world))]
        gathered.append(torch.cat(parts).numpy())
    out[rank] = gathered
    dist.destroy_process_group()


def test_two_gloo_ranks_sharded_by_sequence_equal_one_rank():
    oracle.build()
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    w = wl.make_workload(wl.dataclasses.replace(wl.SPECS[3], B=5, H=2, dk=32, dv=16, N=12))
    full = _oracle_block(w)
    for r in range(world):
        for got, want in zip(res[r], full):
            assert got.shape == want.shape
            assert np.array_equal(got, want)          # bit-identical: same per-sequence arithmetic


def test_gpus_flag_relaunches_or_refuses(monkeypatch):
    import bench
    cmd = bench.launcher_command(["--gpus", "4", "--steps", "2"], 4, 29555)
    assert cmd[1:3] == ["-m", "torch.distributed.run"]
    assert "--nproc-per-node" in cmd and cmd[cmd.index("--nproc-per-node") + 1] == "4"
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert cmd[-4:] == ["--gpus", "4", "--steps", "2"]

    class A:
        gpus = 1
    assert bench.check_world(A, 1) is None               # matching world: run here
    A.gpus = 2
    assert bench.check_world(A, 4) == 2                  # launched with another world size: refuse
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(torch.cuda, "device_count", lambda: 1)
    assert bench.check_world(A, 1) == 2                  # asks for more GPUs than are visible: refuse
