"""The multi-GPU path is independent replicas (no collective on the data
path); the only cross-rank step is the timing reduction of bench.py.  It is
checked here with two gloo ranks on CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = 10.0 * (rank + 1)  # rank 1 is the slow replica
    ms_step, us_block = bench.job_timing(local, steps=5, world=world, dist=dist)
    results[rank] = (ms_step, us_block)
    dist.destroy_process_group()


def test_job_timing_takes_the_slowest_rank_and_divides_by_replicas():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
        got = dict(results)
    # max over ranks = 20 ms for 5 steps = 4 ms per step; 2 replicas
    for rank in range(world):
        ms_step, us_block = got[rank]
        assert ms_step == pytest.approx(4.0)
        assert us_block == pytest.approx(4.0 * 1e3 / world)


def test_job_timing_single_process():
    import bench
    ms_step, us_block = bench.job_timing(12.0, steps=4, world=1)
    assert ms_step == pytest.approx(3.0) and us_block == pytest.approx(3000.0)
