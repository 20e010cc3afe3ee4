"""The benchmark's multi-rank plumbing on CPU: two gloo ranks on 127.0.0.1.
Requests are independent, so N GPUs run N replicas (weak scaling) and the
only cross-rank steps are measurement: the slowest rank's times and the job's
whole throughput.  The reference arm runs on rank 0 only."""
from __future__ import annotations

import importlib.util
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    b = _bench()
    times = b._max_over_ranks([10.0 + rank, 3.0 * (world - rank)], torch.device("cpu"))
    out[rank] = times + [b._job_value(world, 256, times[0])]
    torch.distributed.barrier()
    torch.distributed.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_the_whole_job():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    for r in range(world):
        ms, other, value = out[r]
        assert ms == 11.0 and other == 6.0          # max over ranks of each timing
        assert value == pytest.approx(2 * 256 / 11e-3)  # both ranks' units over the slowest time


def test_single_rank_is_a_no_op(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "1")
    b = _bench()
    assert b._max_over_ranks([1.5, 2.5], torch.device("cpu")) == [1.5, 2.5]
    assert b._job_value(1, 256, 2.0) == pytest.approx(128000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    b = _bench()

    class A:
        steps, warmup = 1, 0
    assert b.run_reference(A()) == 0
    assert capsys.readouterr().out == ""
