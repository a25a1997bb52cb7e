"""The multi-process side of bench.py, on CPU with the gloo backend
(world_size 2, rendezvous on 127.0.0.1): every rank is an independent
replica; the step time is the maximum over ranks and the whole-job value is
the tokens of all ranks over that time; the reference arm works on rank 0
only."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        local = [1.0 + rank, 10.0 - rank]  # rank-dependent step and decode times (ms)
        step_ms, dec_ms = bench.max_over_ranks(dist, world, local, "cpu")
        value = bench.whole_job_tokens_per_s(world, 8192, step_ms)
        dist.barrier()
        out[rank] = (step_ms, dec_ms, value)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo():
    world = 2
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for rank in range(world):
        step_ms, dec_ms, value = out[rank]
        assert step_ms == 2.0          # the slower rank's step time
        assert dec_ms == 10.0
        assert value == pytest.approx(2 * 8192 / 2e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 1, [3.0, 4.0], "cpu") == [3.0, 4.0]
    assert bench.whole_job_tokens_per_s(1, 8192, 0.5) == pytest.approx(8192 / 5e-4)


def test_reference_arm_is_rank_zero_only(monkeypatch, capsys):
    """Under torchrun every rank but 0 leaves the reference arm at once,
    without work or output."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup = 1, 3

    assert bench.reference_arm(A()) is None
    assert capsys.readouterr().out == ""
