"""Multi-rank bench logic on CPU (gloo, world size 2): the step time is the
slowest rank's, the value is the whole-job aggregate, and only rank 0 prints.
The path shards as replicas only, so no collective touches the data path."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], dist)
        out[rank] = (ms, bench.whole_job_tflops(1e12, ms, world), bench.dist_env())
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    times = [3.0, 5.0]
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), times, out), nprocs=world, join=True)
    for r in range(world):
        ms, tflops, env = out[r]
        assert ms == 5.0  # slowest rank
        assert tflops == pytest.approx(2 * 1e12 / 5e-3 / 1e12)
        assert env == (2, r, 0)


def test_single_process_passthrough():
    assert bench.max_over_ranks(4.25) == 4.25
    assert bench.whole_job_tflops(2e12, 1.0, 1) == pytest.approx(2000.0)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class Args:
        workload = "720p"
        steps = 1
        warmup = 0
    assert bench.run_reference(Args()) is None


def test_clock_summary_reads_reasons_and_loaded_median():
    lines = "\n".join([
        "0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2070, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 345, 2070, 120.0, 0x1, Not Active, Not Active, Not Active, Not Active",  # idle sample
    ])
    c = bench.ClockSampler.summarize(lines)
    assert c["sm_max_mhz"] == 2070.0
    assert c["sm_mhz"] == 2070.0  # median of the three loaded samples; the idle one is dropped
    assert c["reasons"] == ["sw_power_cap"]
    assert not (bench.THROTTLE_REASONS & set(c["reasons"]))  # power capping keeps the run
    hot = bench.ClockSampler.summarize("0, 1500, 2070, 1400.0, 0x40, Not Active, Active, Not Active, Not Active")
    assert bench.THROTTLE_REASONS & set(hot["reasons"]) == {"hw_thermal_slowdown"}  # measured again


def test_workload_config_names_the_workload():
    import wsa_inputs
    wl = wsa_inputs.WORKLOADS["720p"]
    c = bench.workload_config(wl, (6, 15, 27), [36, 64])
    assert c["tokens"] == 75600 and c["heads"] == 24 and c["head_dim"] == 128 and c["windows"] == [36, 64]
    assert c["workload"].startswith("720p: T=21,H=45,W=80 (75600 tokens)")
    assert "wt,wh,ww=6,15,27" in c["workload"] and "gathers/scatters through ids" in c["workload"]
    assert "plan-packed order" in bench.workload_config(wl, (6, 15, 27), [36, 64], packed=True)["workload"]
    assert c["parallelism"] == "single" and bench.workload_config(wl, (6, 15, 27), [36, 64], ws=2)["parallelism"] == "replicas"
