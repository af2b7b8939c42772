"""The benchmark's multi-rank host logic on CPU: two gloo ranks, each timing its own
independent decode problem; the job's step time (the value) is the max over ranks, a
latency that replicas do not shorten, and the job's aggregate steps per second is the rank
count over that time (weak scaling, no data-path collective)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        assert (w, r, local) == (world, rank, rank)
        step_ms = 0.050 + 0.010 * rank          # rank 1 is the slower one
        worst = bench.reduce_max(step_ms, world)
        bench.barrier(world)
        out[rank] = (worst, bench.job_value(worst, world), bench.job_steps_per_s(worst, world))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_and_job_value():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    for rank in range(world):
        worst, value, steps_per_s = out[rank]
        assert worst == pytest.approx(0.060)
        assert value == pytest.approx(60.0)  # µs per step: the slowest rank's, not divided
        assert steps_per_s == pytest.approx(2 / 0.060e-3)


def test_single_rank_is_plain():
    import bench
    assert bench.reduce_max(1.25, 1) == 1.25
    assert bench.job_value(0.1, 1) == pytest.approx(100.0)
    assert bench.job_steps_per_s(0.1, 1) == pytest.approx(10000.0)


def test_reference_arm_runs_on_rank_zero_only(capsys, monkeypatch):
    """The reference arm (the CPU oracle) prints one JSON line on rank 0 and nothing on the
    other ranks, with the main arm's metric, unit and workload text."""
    import argparse
    import json

    import bench
    from kv_cache_int8_gb300 import workloads as W
    monkeypatch.setenv("HSA_REF_BUDGET_S", "0.5")
    args = argparse.Namespace(config="tiny-8k", steps=2, warmup=0, gpus=2)
    assert bench.run_reference(args, 2, 1) == 0
    assert capsys.readouterr().out == ""
    assert bench.run_reference(args, 2, 0) == 0
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "us/step" and line["higher_is_better"] is False
    assert line["config"]["workload"] == bench.workload_text(W.CONFIGS["tiny-8k"])
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
