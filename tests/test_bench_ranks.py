"""Multi-rank host logic of the benchmark, on CPU with the gloo backend.

With N > 1 every rank runs its own copy of the workload; the job's rate is
the units of all ranks over the slowest rank's time.  Two gloo ranks check
that reduction and that a step count mismatch cannot inflate the rate.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    secs = [2.0, 3.0][rank]          # the second rank is slower
    units = [100.0, 140.0][rank]     # and did more work
    rate, slowest = bench.job_rate(secs, units, world, "cpu")
    q.put((rank, rate, slowest))
    dist.destroy_process_group()


def test_job_rate_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, rate, slowest in got:
        assert slowest == 3.0
        assert rate == pytest.approx(240.0 / 3.0)


def test_job_rate_single_rank():
    import bench
    assert bench.job_rate(2.0, 10.0, 1) == (5.0, 2.0)
