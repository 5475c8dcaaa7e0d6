"""The multi-rank host logic of bench.py on CPU: two gloo ranks (one replica of
the workload per rank, no data-path collective) agree on the slowest rank's time
and report whole-job throughput; the reference arm runs on rank 0 only."""
import argparse
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        dist.barrier()
        slowest = bench.max_over_ranks(times[rank], dist, "cpu")
        value = bench.job_value(1.0e12, world, slowest)
        out.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(0.5, 0.75), (2.0, 1.0)])
def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_work(times):
    ctx = mp.get_context("spawn")
    out = ctx.SimpleQueue()
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, times, out), nprocs=2, join=True,
                       start_method="spawn")
    got = sorted(out.get() for _ in range(2))
    assert [g[0] for g in got] == [0, 1]
    slow = max(times)
    for _, s, v in got:
        assert s == slow                       # both ranks agree on the slowest rank
        assert v == pytest.approx(2 * 1.0e12 / slow)  # weak scaling: the work of both ranks


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.25) == 0.25
    assert bench.job_value(3.0, 1, 2.0) == 1.5


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench
    import synth
    args = argparse.Namespace(steps=1, warmup=0, gpus=2, dropout=0.0)
    assert bench.run_reference(args, synth.WORKLOADS["fp32_n256"], rank=1) is None
    assert capsys.readouterr().out == ""


def test_fp8_reference_arm_line(capsys):
    """bench.py --fp8 --impl reference: rank 0 times the oracle's FP8 path and prints one
    line with the contract's keys; another rank prints nothing."""
    sys.path.insert(0, ROOT)
    import json

    import bench
    import synth
    w = synth.Workload("fp8_small", 1, 2, 256, 64, "bf16", 3, causal=(False, True))
    args = argparse.Namespace(steps=1, warmup=0, gpus=1, impl="reference", fp8=True)
    bench.run_fp8(args, w, rank=1, world=2, local=1)
    assert capsys.readouterr().out == ""
    bench.run_fp8(args, w, rank=0, world=1, local=0)
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["metric"] == bench.FP8_METRIC
    assert line["value"] > 0 and line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["config"]["causal"] == [False, True]
