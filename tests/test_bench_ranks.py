"""The multi-rank bookkeeping of bench.py, on CPU with two gloo ranks.

Under torchrun every rank times its own replica of the workload (weak
scaling, no collective on the data path); the job's time is the slowest
rank's, taken with one MAX all-reduce, and the job's value counts every
rank's FLOPs.  These tests run that code as two processes on the host.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        slowest = bench.slowest_rank_ms(times[rank], world, "cpu")
        dist.barrier()
        out[rank] = slowest
    finally:
        dist.destroy_process_group()


def test_slowest_rank_time_is_the_maximum_on_every_rank():
    times = [12.5, 20.25]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(2, _free_port(), times, out), nprocs=2, join=True)
        got = dict(out)
    assert got == {0: 20.25, 1: 20.25}


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_ms(7.0, 1, "cpu") == 7.0


def _value_main(rank, world, port, flops, times, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.slowest_rank_ms(times[rank], world, "cpu")
        out[rank] = bench.job_tflops_sum(flops[rank], ms, world, "cpu")
    finally:
        dist.destroy_process_group()


def test_job_value_sums_unequal_rank_work_over_the_slowest_time():
    # rank 0: 1e12 FLOPs in 0.4 ms, rank 1: 3e12 FLOPs in 0.5 ms -> the job
    # moved 4e12 FLOPs in 0.5 ms (the slowest rank): 8000 TFLOP/s, on both ranks
    flops, times = [1e12, 3e12], [0.4, 0.5]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_value_main, args=(2, _free_port(), flops, times, out), nprocs=2, join=True)
        got = dict(out)
    assert got[0] == pytest.approx(8000.0) and got[1] == pytest.approx(8000.0)


def test_job_value_of_one_rank():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_tflops_sum(1e12, 0.5, 1, "cpu") == pytest.approx(2000.0)


def test_replicas_share_their_shapes():
    # under torchrun every rank draws its own values but the same window
    # lengths, so the job's FLOPs are the same on every rank
    import sys
    sys.path.insert(0, ROOT)
    import synth
    w0 = synth.workload("varlen8", seed=0, shape_seed=0)
    w3 = synth.workload("varlen8", seed=3, shape_seed=0)
    assert w0.lp == w3.lp and w0.lc == w3.lc
    a, b = synth.make_inputs(w0), synth.make_inputs(w3)
    assert a["q"].shape == b["q"].shape and not bool((a["q"] == b["q"]).all())
