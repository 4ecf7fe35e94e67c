"""Multi-rank logic of bench.py on CPU (gloo, world size 2).

The path runs as independent replicas (one batch per GPU, no collective on the
data path); only the timing is reduced across ranks, and the reference arm runs
on rank 0 alone. These tests exercise exactly that host-side logic.
"""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.rank_env()
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank)  # rank 1 is slower
        out[rank] = (w, r, local, slowest, bench.rank_seed(7, r))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_per_rank_batches():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][:3] == (2, 0, 0) and res[1][:3] == (2, 1, 1)
    assert res[0][3] == res[1][3] == 15.0          # both ranks report the slowest time
    assert res[0][4] != res[1][4]                  # each replica draws its own batch


def test_max_over_ranks_without_process_group():
    assert bench.max_over_ranks(3.5) == 3.5


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    import argparse

    ns = argparse.Namespace(workload="tiny", seed=0, steps=1, warmup=0, gpus=2)
    bench.run_reference(ns)  # returns at once on rank 1
    assert capsys.readouterr().out == ""
