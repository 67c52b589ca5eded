"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

The heads of a problem are independent (K mean, scales and attention are
per (b, h)), so ranks either split the heads of one problem or run replicas,
with no data-path collective; the only cross-rank step is taking the slowest
rank's time.  These tests check the head bookkeeping (every head computed
exactly once) and the timing reduction.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank            # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms, world)
        out[rank] = (ms, bench.whole_job_tops(1_000_000_000_000, world, ms))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_rank():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    # 2 replicas x 1e12 ops in 15 ms
    assert res[0][1] == pytest.approx(2e12 / 15e-3 / 1e12)


def _split_worker(rank, world, port, H, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = bench.head_range(rank, world, H)
        ranges = [None] * world
        dist.all_gather_object(ranges, mine)
        ms = bench.max_over_ranks(20.0 - 4.0 * rank, world)
        out[rank] = (ranges, ms)
    finally:
        dist.destroy_process_group()


def test_two_rank_head_split_computes_every_head_once():
    world, H = 2, 24
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_split_worker, args=(world, port, H, out), nprocs=world, join=True)
        res = dict(out)
    ranges = res[0][0]
    assert ranges == res[1][0]
    covered = [h for h0, h1 in ranges for h in range(h0, h1)]
    assert sorted(covered) == list(range(H))          # each head exactly once
    assert res[0][1] == res[1][1] == 20.0


def test_head_ranges_partition_the_heads():
    import bench
    for H in range(1, 41):
        for world in range(1, min(H, 8) + 1):
            ranges = [bench.head_range(r, world, H) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == H
            assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))     # contiguous, disjoint
            sizes = [h1 - h0 for h0, h1 in ranges]
            assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1
    with pytest.raises(ValueError):
        bench.head_range(0, 25, 24)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_tops(3_298_534_883_328, 1, 3.48) == pytest.approx(947.856, rel=1e-4)
