"""The host side of bench.py's multi-process launch, on CPU with two gloo ranks.

The projection does not shard across GPUs here: each rank runs an independent
replica of the whole step, so the only cross-rank logic is the timing
reduction (the slowest rank's time), the whole-job rate (every rank's work over
that time) and which rank reports.  These run as two processes on 127.0.0.1.
"""
import json
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, _ = bench.dist_env()
        # each replica's own step time: rank 1 is the slow one
        t = 0.010 * (1 + r)
        slowest = bench.max_over_ranks(t, dist, "cpu")
        rate = bench.job_throughput(w, 5.0e12, slowest)
        with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
            json.dump({"rank": r, "world": w, "slowest": slowest, "rate": rate}, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn",
                       join=True)
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for g in got:
        assert g["world"] == world
        assert g["slowest"] == pytest.approx(0.020)  # every rank sees the max
        assert g["rate"] == pytest.approx(world * 5.0e12 / 0.020)  # all ranks' work over the max


def test_single_process_needs_no_group():
    import bench

    assert bench.max_over_ranks(0.25, None, "cpu") == 0.25
    assert bench.job_throughput(1, 3.0, 1.5) == 2.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    # under torchrun every rank but 0 leaves at once, printing nothing
    import bench

    import argparse

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(gpus=2, steps=1, warmup=0, impl="reference", no_cpu_baseline=True)
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""
