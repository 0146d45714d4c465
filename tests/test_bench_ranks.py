"""Multi-rank bench logic on CPU: two gloo ranks run the aggregation `bench.py` uses for
--gpus N (replicas: each rank times its own step; the job time is the slowest rank's and
the job rate counts every rank's work)."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, l = bench.dist_setup(None)
        ms = 10.0 + 5.0 * rank                       # rank 1 is the slow one
        job_ms = bench.max_over_ranks(torch, ms, "cpu", w)
        out[rank] = (w, r, l, job_ms, bench.job_throughput(100.0, w, job_ms))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_all_work():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        w, r, l, job_ms, rate = res[rank]
        assert (w, r, l) == (2, rank, rank)
        assert job_ms == 15.0                         # max over ranks
        assert rate == pytest.approx(100.0 * 2 / 15e-3)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(torch, 7.5, "cpu", 1) == 7.5
    assert bench.job_throughput(3.0, 1, 2.0) == pytest.approx(1500.0)


def test_reference_arm_runs_on_rank_zero_only():
    import bench
    # ranks other than 0 leave at once, without touching the oracle or the GPU
    assert bench.reference_main(None, 2, 1) == 0
