"""The N > 1 benchmark path on CPU: two gloo ranks run independent replicas and
agree on the slowest rank's step time; the job throughput counts every rank's
bytes over that time.  No data-path collective exists on the path itself."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, results):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [1.5, 2.25][rank]          # rank 1 is the slow replica
        results[rank] = bench.max_over_ranks(ms, world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(results) == {0: 2.25, 1: 2.25}


def test_job_throughput_counts_every_replica():
    one = bench.job_throughput_gbs(565_350_400, 1, 0.0933)
    two = bench.job_throughput_gbs(565_350_400, 2, 0.0933)
    assert two == pytest.approx(2 * one)
    assert one == pytest.approx(565_350_400 / 93.3e-6 / 1e9)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.0, 1) == 3.0
