"""The multi-rank logic of bench.py on CPU with gloo, world size 2.

Under torchrun every rank runs its own replica of the workload (the (batch,
head) units are independent, so no collective sits on the data path); the
ranks meet only to take the slowest rank's time, and rank 0 alone prints.
These tests run that logic in two CPU processes over gloo; no GPU is used.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # per-rank step, attention and prologue times: rank 1 is slower in two of them
        mine = [1.0 + rank, 0.5 + 0.25 * rank, 0.2 - 0.1 * rank]
        got = bench.max_over_ranks(mine, world, dist, torch, "cpu")
        assert bench.dist_env() == (rank, world, rank)
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_slowest_rank_decides_over_gloo():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for rank in range(world):
        assert out[rank] == pytest.approx([2.0, 0.75, 0.2])


def test_job_throughput_counts_every_replica():
    # 260.9 GFLOP per rank in 0.2 ms on each of 4 ranks = 4 x 1304.6 TFLOP/s
    assert bench.job_throughput(260.9e9, 4, 0.2) == pytest.approx(4 * 1304.5, rel=1e-3)
    assert bench.job_throughput(260.9e9, 1, 0.2) == pytest.approx(1304.5, rel=1e-3)


def test_single_rank_reduction_is_the_identity():
    assert bench.max_over_ranks([3.0, 1.5], 1, None, torch, "cpu") == [3.0, 1.5]


def _reference_rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import io
    import contextlib

    class Args:
        workload = "tiny_320"
        reference_rows = 64
        steps = 1
        warmup = 3
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(Args)
    out[rank] = buf.getvalue()


def test_reference_arm_prints_on_rank_zero_only():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_reference_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    import json
    line = json.loads(out[0])
    assert line["impl"] == "reference" and line["n_gpus"] == world
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert out[1] == ""
