"""Host logic of the multi-GPU bench path (independent replicas), run as
world-size-2 gloo ranks on the CPU: the whole-job time is the slowest rank's,
the committed tokens are every rank's, and only rank 0 runs the reference arm."""
import io
import os
import contextlib
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = bench.dist_env()
        ms, committed = bench.reduce_over_ranks(10.0 + 3.0 * rank, 5 * (rank + 1), w, "cpu")
        out[rank] = (r, lr, w, ms, committed)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_time_by_max_and_tokens_by_sum():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    for rank in range(world):
        r, lr, w, ms, committed = out[rank]
        assert (r, lr, w) == (rank, rank, world)
        assert ms == 13.0          # the slowest rank
        assert committed == 15     # 5 + 10


def test_single_rank_is_unchanged():
    assert bench.reduce_over_ranks(7.5, 3, 1, "cpu") == (7.5, 3)


def test_reference_arm_runs_on_rank_0_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        workload = "full_stack"
        steps = 1
        warmup = 0
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert bench.run_reference(Args()) is None
    assert buf.getvalue() == ""  # the other ranks exit without work or output
