"""The multi-GPU path is replicas only (slots and heads are independent; there
is no exchange step).  What the ranks share is the bench's aggregation: the
job clock is the slowest rank and throughput counts every rank's work.  That
logic is exercised here with world_size-2 gloo process groups on CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dt = bench.max_over_ranks(times[rank])
        out[rank] = (dt, bench.job_throughput(16, 100, world, dt))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    world, port = 2, _free_port()
    times = [0.010, 0.014]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        assert res[r][0] == pytest.approx(0.014)
        assert res[r][1] == pytest.approx(16 * 100 * 2 / 0.014)


def test_single_process_is_identity():
    assert bench.max_over_ranks(0.25) == 0.25
    assert bench.job_throughput(16, 10, 1, 2.0) == 80.0
