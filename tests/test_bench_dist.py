"""The multi-rank host logic of bench.py, on CPU with two gloo ranks.

bench.py runs one independent replica of the step per GPU (the path has no
exchange step): the only collectives are the barrier around the timed region
and the max over ranks of its wall time.  These tests start two processes on
127.0.0.1, go through bench.py's own rendezvous (dist_setup reads RANK,
WORLD_SIZE, LOCAL_RANK and MASTER_* from the environment), and check that
every rank ends with the slowest rank's time and the whole-job value, and
that the reference arm does its work on rank 0 only.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import sys
    sys.path.insert(0, ROOT)
    import bench
    r, w, local = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    # rank r "measured" 10 + 5r ms for 4 steps whose roofline time is 1 ms each
    ms_total, ms_step, value = bench.job_value(10.0 + 5.0 * r, 4, 1e-3, w)
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    results[rank] = (ms_total, ms_step, value)


def test_two_ranks_report_the_slowest_rank_and_the_whole_job_value():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.start_processes(_rank_main, args=(world, port, results), nprocs=world,
                           start_method="spawn", join=True)
        got = dict(results)
    slowest = 10.0 + 5.0 * (world - 1)
    for r in range(world):
        ms_total, ms_step, value = got[r]
        assert ms_total == pytest.approx(slowest)
        assert ms_step == pytest.approx(slowest / 4)
        # both ranks did 4 steps of 1 ms roofline work each: 8 ms of roofline time
        assert value == pytest.approx(100.0 * world * 1e-3 / (slowest / 4 * 1e-3))


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
    ms_total, ms_step, value = bench.job_value(20.0, 10, 1e-3, 1)
    assert (ms_total, ms_step) == (20.0, 2.0)
    assert value == pytest.approx(50.0)


def _reference_rank(rank, world, port, results):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import sys
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        steps, warmup, gpus = 1, 0, world

    if rank == 0:
        results[rank] = "skipped"  # rank 0 would time the oracle: not repeated here
        return
    bench.bench_reference(Args())  # the other ranks must return at once, without work
    results[rank] = "returned"


def test_reference_arm_runs_on_rank_zero_only():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.start_processes(_reference_rank, args=(world, port, results), nprocs=world,
                           start_method="spawn", join=True)
        assert dict(results) == {0: "skipped", 1: "returned"}
