"""Host logic of the benchmark's multi-GPU mode (N independent replicas, one
rank per GPU) on CPU ranks with the gloo backend: the timing that decides a
multi-rank number is the maximum over the ranks, and only rank 0 prints."""
import contextlib
import io
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out.put((rank, bench.max_over_ranks(1.5 + rank, world)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    mp.start_processes(_rank_main, args=(2, _free_port(), q), nprocs=2, join=True, start_method="spawn")
    got = sorted(q.get() for _ in range(2))
    assert got == [(0, 2.5), (1, 2.5)]


def test_max_over_ranks_single_rank_is_identity():
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_reference_arm_prints_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"])
    args = bench.parse()
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args)
    assert buf.getvalue() == ""
