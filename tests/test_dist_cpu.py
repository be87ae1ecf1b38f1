"""Multi-process path of the benchmark on CPU: two gloo ranks reduce their
step times to the slowest rank's, and the whole-job value counts every
rank's rows.  (The decode path itself has no cross-GPU exchange: ranks are
independent replicas.)"""

import os

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        mine = [1.0 + rank, 10.0 - rank]          # rank 1 slower on the first, faster on the second
        got = bench.max_over_ranks(mine)
        out[rank] = (got, bench.aggregate_value(64, 10, world, got[0]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_slowest():
    if not dist.is_available():
        pytest.skip("torch.distributed unavailable")
    port = 29500 + os.getpid() % 1000
    with mp.get_context("spawn").Manager() as m:     # no fork of a threaded parent
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        got, value = res[rank]
        assert got == [2.0, 10.0]
        assert value == pytest.approx(64 * 10 * 2 / 2.0)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert bench.aggregate_value(64, 5, 1, 2.0) == pytest.approx(160.0)
