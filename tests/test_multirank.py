"""The multi-process path of bench.py on CPU: two gloo ranks (127.0.0.1).

The backward does not shard across GPUs here (independent replicas), so what
is checked is the host logic around it: the barrier, the max-over-ranks time,
the whole-job throughput from it, and that the reference arm runs on rank 0
only (the other ranks exit without work)."""
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
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        bench.barrier(world)
        ms = 1.0 + 2.0 * rank            # rank 1 is the slow one
        m = bench.max_over_ranks(ms, world)
        out[rank] = (m, bench.job_throughput(1000, world, m))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world = 2
    out = mp.get_context("spawn").Manager().dict()   # no fork: the parent may hold threads
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1]
    m, v = out[0]
    assert m == 3.0
    assert v == pytest.approx(2 * 1000 / 3e-3)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert bench.job_throughput(16384, 1, 2.0) == pytest.approx(8.192e6)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert bench.run_reference(bench.parse()) == 0
    assert capsys.readouterr().out == ""
