"""The multi-GPU path is independent replicas (every (b, h_q, Q-tile) unit is independent; no
data-path exchange).  What bench.py adds for N > 1 is host logic: a barrier around the timed
region, the maximum of the per-rank times and the whole-job throughput.  This checks that logic
with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    dist.barrier()
    slowest = bench.max_over_ranks(times[rank])
    out[rank] = (slowest, bench.job_throughput(10.0, world, slowest))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("times", [(2.0, 3.0), (5.0, 1.5)])
def test_two_gloo_ranks_take_the_slowest_time(times):
    ctx = mp.get_context("spawn")
    port = _free_port()
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, times, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        slowest = max(times)
        for r in range(2):
            assert out[r][0] == slowest
            assert out[r][1] == pytest.approx(20.0 / slowest)


def test_single_process_needs_no_group():
    import bench

    assert bench.max_over_ranks(4.25) == 4.25
    assert bench.job_throughput(8.0, 1, 2.0) == 4.0
