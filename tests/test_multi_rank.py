"""The multi-rank host logic of bench.py with two gloo processes on the CPU:
the job's time is the slowest rank's, and the whole-job rate counts every
rank's units (weak scaling, one replica per rank)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 7.5 * rank                 # rank 1 is the slower one
        results[rank] = bench.max_over_ranks(mine, world, "cpu")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        assert dict(results) == {0: 17.5, 1: 17.5}


def test_whole_job_rate_is_weak_scaling():
    import bench
    one = bench.whole_job_rate(471064576, 1, 100, 9.0)
    two = bench.whole_job_rate(471064576, 2, 100, 9.0)
    assert two == pytest.approx(2 * one)
    assert bench.max_over_ranks(3.0, 1) == 3.0
