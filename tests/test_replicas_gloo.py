"""Multi-process (N > 1) path of bench.py on CPU: world_size-2 gloo ranks.

The decode step does not shard, so N GPUs run N independent replicas; the
only cross-rank step is the timing aggregation (max over ranks of the time,
sum of the ranks' steps), and the reference arm runs on rank 0 alone."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, steps, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        v = bench.replica_throughput(times[rank], steps, dist, device="cpu")
        out[rank] = v
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(2.0, 3.0), (5.0, 1.0)])
def test_replica_throughput_two_gloo_ranks(times):
    world, steps = 2, 10
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), times, steps, out), nprocs=world,
                       join=True, start_method="spawn")
    expect = world * steps / max(times)
    assert out[0] == pytest.approx(expect) and out[1] == pytest.approx(expect)


def test_replica_throughput_single_process():
    assert bench.replica_throughput(2.0, 10, None) == pytest.approx(5.0)


def test_reference_arm_other_ranks_do_nothing(capsys):
    class A:
        model = "qwen2.5-7b"
        context = 2048
    bench.run_reference(A(), rank=1, world=2)
    assert capsys.readouterr().out == ""


def test_reference_arm_runs_the_requested_steps(capsys):
    """Rank 0 of the reference arm times W untimed and exactly K timed whole
    oracle decode steps and prints one JSON line whose ms_per_step * steps
    is the timed wall time."""
    import json

    class A:
        model = "qwen2.5-0.5b"
        context = 64
        steps = 2
        warmup = 1
        gpus = 1
    bench.run_reference(A(), rank=0, world=1)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 1
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert "1 untimed, 2 timed" in line["cpu_baseline"]["sample"]
    assert line["cpu_baseline"]["cpu_model"]
    assert abs(line["ms_per_step"] * line["steps"] / 1e3 - line["steps"] / line["value"]) < 1e-6
