"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

The attention path shards into independent problems, so ranks run replicas
with no data-path collective; the only cross-rank step is taking the slowest
rank's time and counting every rank's work.
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


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_tops(3_298_534_883_328, 1, 3.48) == pytest.approx(947.856, rel=1e-4)
