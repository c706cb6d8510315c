"""The replica (N > 1) path of bench.py on CPU: world size 2 over gloo.

The layer does not shard (one process per GPU runs a full replica on its own
tokens), so the only cross-rank steps are the barriers and the maximum of the
per-rank timings; these tests run them over a gloo process group on the host,
plus the whole-job throughput formula and the per-rank input seeds."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from sparse_mixture_experts_52_b300 import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [10.0 + rank, 5.0 - rank, 7.0 * (rank + 1)]
        dist.barrier()
        got = bench.max_over_ranks(mine, world, torch.device("cpu"))
        # inputs of replica r are drawn from seed + r: the replicas differ
        cfg = synth.workload("tiny_fp32_top2", T=32)
        x = synth.make_inputs(cfg, device="cpu", seed=cfg["seed"] + rank)["x"]
        xs = [torch.empty_like(x) for _ in range(world)]
        dist.all_gather(xs, x)
        out[rank] = (got, bool(torch.equal(xs[0], xs[1])))
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_take_the_slowest_rank():
    world = 2
    with mp.get_context("spawn").Manager() as m:   # no fork of this (threaded) process
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                           start_method="spawn")
        res = dict(out)
    for r in range(world):
        got, same_inputs = res[r]
        assert got == [11.0, 5.0, 14.0], got
        assert not same_inputs


def test_single_process_keeps_its_own_timings():
    assert bench.max_over_ranks([1.5, 2.5], 1, torch.device("cpu")) == [1.5, 2.5]


def test_whole_job_throughput_is_weak_scaling():
    # 2 replicas x 4096 tokens x 10 steps in 5 ms of the slowest replica
    assert bench.whole_job_tokens_per_s(4096, 2, 10, 5.0) == pytest.approx(2 * 4096 * 10 / 0.005)
    assert bench.whole_job_tokens_per_s(4096, 1, 10, 5.0) == pytest.approx(4096 * 10 / 0.005)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    class A:
        workload = "tiny_fp32_top2"
        steps = 1
        warmup = 0
        cpu_rows = 8
    bench.run_reference(A(), rank=1, world=2)   # rank 1: no work, no output
    assert capsys.readouterr().out == ""
