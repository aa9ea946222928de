"""The multi-GPU path of the benchmark on CPU: world_size-2 gloo ranks.

The hot path shards by (sequence, KV head) with no exchange step, so N GPUs
run N independent replicas; the only cross-rank steps are the barrier around
the timed region and the maximum of the timings over ranks, which rank 0
reports. These tests run that host logic on two CPU processes (gloo backend,
rendezvous on 127.0.0.1) and check the rank/world parsing and the reference
arm's rank-0-only behaviour.
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        dist.barrier()
        # each rank "timed" a different duration; every rank gets the maximum
        mine = [10.0 + rank, 5.0 - rank, 7.5 * (rank + 1)]
        got = bench.max_over_ranks(mine, world)
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:   # no fork of a threaded process
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    expect = [11.0, 5.0, 15.0]
    assert res[0] == expect and res[1] == expect


def test_max_over_ranks_single_rank_is_identity():
    assert bench.max_over_ranks([3.0, 1.5], 1) == [3.0, 1.5]


def test_reference_arm_only_rank0_works(monkeypatch):
    # under torchrun the reference arm runs on rank 0 only; other ranks exit
    # without work (run_reference returns None before touching any device)
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class Args:
        steps, warmup = 1, 0

    assert bench.run_reference(Args()) is None


def test_dist_env_defaults(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
