"""The N > 1 bench path runs independent replicas: each rank times its own
copy of the workload, the job's time is the slowest rank's (MAX all-reduce),
and the value is every rank's FLOP over that time.  Checked with world size 2
on the gloo backend on CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, ret):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [120.0, 150.0][rank]
    slowest = bench.max_over_ranks(ms, dist, "cpu")
    ret[rank] = (slowest, bench.job_tflops(world, bench.STEP_FLOP, slowest))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_report_max_time_and_job_throughput():
    import bench

    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    ret = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, ret)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        slowest, tflops = ret[r]
        assert slowest == 150.0
        assert tflops == pytest.approx(2 * bench.STEP_FLOP / 0.150 / 1e12)


def test_single_rank_helpers():
    import bench

    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.job_tflops(1, 1e12, 1000.0) == pytest.approx(1.0)
