"""Multi-rank host logic of bench.py on CPU: two gloo ranks, the whole-job
rate (units of all ranks over the slowest rank's time) and the max over ranks."""
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

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    seconds = [1.0, 2.0][rank]
    rate = bench.whole_job_rate(10.0, seconds, dist)
    worst = bench.max_over_ranks(seconds, dist)
    bench.barrier(dist)
    dist.destroy_process_group()
    out[rank] = (rate, worst)


def test_two_rank_aggregation():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        rate, worst = res[rank]
        assert worst == 2.0
        assert rate == pytest.approx(20.0 / 2.0)


def test_single_rank_is_identity():
    import bench

    assert bench.whole_job_rate(10.0, 2.0, None) == 5.0
    assert bench.max_over_ranks(3.0, None) == 3.0
