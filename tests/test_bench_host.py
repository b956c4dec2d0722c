"""Host logic of bench.py that needs no GPU: the multi-rank aggregation (two
gloo ranks on CPU), the whole-job value and the clock-record summary."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(torch, times[rank], "cpu", world)
        out[rank] = got
    finally:
        torch.distributed.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world, times = 2, [0.125, 0.5]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), times, out), nprocs=world, join=True)
        res = dict(out)
    # every rank reports the slowest rank's time
    assert res == {0: 0.5, 1: 0.5}


def test_max_over_ranks_single_rank_is_identity():
    assert bench.max_over_ranks(torch, 0.25, "cpu", 1) == 0.25


def test_job_value_is_weak_scaling_aggregate():
    flops = 2.0 * 8192 * 2048 * 6144
    one = bench.job_value(1, flops, 0.11)
    assert one == pytest.approx(flops / 0.11e-3 / 1e12)
    # N replicas of the same step in the same time: N times the job throughput
    assert bench.job_value(4, flops, 0.11) == pytest.approx(4 * one)
    # a slower slowest rank lowers the whole job's figure
    assert bench.job_value(4, flops, 0.22) == pytest.approx(2 * one)


def test_clock_summary_reasons_and_median():
    c = bench.ClockSampler(0)
    c.lines = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1395.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2055, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    s = c.summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2055
    assert s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    c.lines = ["0, 1500, 2070, 1400, 0x40, Not Active, Active, Not Active, Not Active"]
    assert bench.ClockSampler.summary(c)["reasons"] == ["hw_thermal_slowdown"]
