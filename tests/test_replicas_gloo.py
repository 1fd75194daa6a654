"""The multi-GPU path is replicas only (the product shards by columns with no exchange), so
what runs on several ranks is the benchmark's host logic: the barrier around the timed
region, the max over ranks of the step time, and rank 0 alone running the reference arm.
These run here as two gloo ranks on the CPU."""
from __future__ import annotations

import argparse
import io
import os
import socket
import contextlib

import pytest


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench._DIST.update(on=True, device="cpu")
        bench.barrier()
        mine = 1.5 + 2.0 * rank  # this rank's step time
        out[rank] = bench.max_over_ranks(mine)
        bench.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_barrier_with_two_gloo_ranks():
    import torch.multiprocessing as mp
    port = _free_port()
    with mp.Manager() as manager:
        out = manager.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        assert dict(out) == {0: 3.5, 1: 3.5}  # both ranks see the slowest rank's time


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import bench
    args = argparse.Namespace(steps=1, warmup=0, gpus=2)
    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args)
    assert buf.getvalue() == ""  # no work, no line on rank 1
