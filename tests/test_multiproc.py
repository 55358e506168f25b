"""bench.py's multi-rank bookkeeping on the CPU with two gloo ranks.

With N > 1 every rank runs its own replica of the workload (weak scaling,
no collective on the data path); the whole-job number is the bytes of all
ranks over the slowest rank's time, and the timed region is bracketed by
barriers. This checks that arithmetic with world_size 2 over gloo.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    d = bench.dist_init(world, "gloo")
    assert d is not None
    bench.barrier(d)
    seconds = 1.0 + rank          # rank 1 is the slower one
    units = 100.0 * (rank + 1)    # bytes each rank processed
    t, u = bench.aggregate(d, seconds, units)
    out[rank] = (t, u)
    bench.barrier(d)
    d.destroy_process_group()


def test_two_gloo_ranks_aggregate_max_time_and_total_bytes():
    port = _free_port()
    manager = mp.get_context("spawn").Manager()   # no fork of this (threaded) process
    out = manager.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1] == (2.0, 300.0)


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_init(1, "gloo") is None
    assert bench.aggregate(None, 1.5, 42.0) == (1.5, 42.0)
