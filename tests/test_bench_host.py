"""Host logic of bench.py that needs no GPU: the multi-rank aggregation (two
gloo ranks on CPU), the whole-job value, the clock-record summary and the
reference arm (the oracle on the host cores)."""
import json
import os
import socket
import subprocess
import sys

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


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run_reference(env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--steps", "1", "--warmup", "0"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_contract_line():
    r = _run_reference({"RANK": "0", "WORLD_SIZE": "1"})
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 1 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] > 0
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"]


def test_reference_arm_other_ranks_exit_quietly():
    r = _run_reference({"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
