"""The multi-process path of bench.py on CPU: two gloo ranks, as torchrun launches them.

The layer itself never exchanges data between ranks (replicas, weak scaling); what
crosses ranks is the timing: the job takes as long as its slowest replica and its
throughput counts every replica's tokens."""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank                     # rank 1 is the slower replica
        total = bench.max_over_ranks(ms, world, "cpu")
        value = bench.job_tokens_per_s(8192, 4, world, total)
        dist.barrier()
        results[rank] = (total, value)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_and_job_throughput_with_gloo(world):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), results), nprocs=world,
                           join=True, start_method="spawn")
        res = dict(results)
    assert sorted(res) == list(range(world))
    slowest = 10.0 + 5.0 * (world - 1)
    for total, value in res.values():
        assert total == slowest                    # every rank sees the slowest time
        assert value == pytest.approx(8192 * 4 * world / (slowest / 1000.0))


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(12.5, 1, "cpu") == 12.5
    assert bench.job_tokens_per_s(100, 2, 1, 1000.0) == pytest.approx(200.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    # torchrun starts every rank; only rank 0 times the oracle and prints its line
    monkeypatch.setenv("RANK", "1")

    class Args:
        warmup, steps, gpus = 0, 1, 2

    from synth import get
    assert bench.run_reference(Args(), get("switch")) == 0
