"""bench.py's multi-rank bookkeeping on the CPU with two gloo ranks.

With N > 1 every rank runs its own replica of the workload (weak scaling,
no collective on the data path); the whole-job number is the bytes of all
ranks over the slowest rank's time, and the timed region is bracketed by
barriers. This checks that arithmetic with world_size 2 over gloo, both
with ranks started here and with ranks that bench.py spawns itself (its
path when --gpus N is given without torch.distributed.run).
"""
import json
import os
import socket
import subprocess
import sys

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


def _spawned_rank(outdir):
    """Runs in each process bench.spawn_replicas starts: the environment it set
    up must carry a gloo rendezvous and the aggregation."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    rank, world, local = bench.dist_env()
    d = bench.dist_init(world, "gloo")
    assert d is not None and d.get_rank() == rank and d.get_world_size() == world
    bench.barrier(d)
    t, u = bench.aggregate(d, 0.5 * (rank + 1), 10.0 * (rank + 1))
    with open(os.path.join(outdir, f"{rank}.json"), "w") as f:
        json.dump({"rank": rank, "local": local, "world": world, "t": t, "u": u}, f)
    bench.barrier(d)
    d.destroy_process_group()


def test_bench_spawns_its_own_replicas(tmp_path):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    rc = bench.spawn_replicas(2, _spawned_rank, str(tmp_path))
    assert rc == 0
    got = [json.load(open(tmp_path / f"{r}.json")) for r in range(2)]
    for r, g in enumerate(got):
        assert g["rank"] == r and g["local"] == r and g["world"] == 2
        assert (g["t"], g["u"]) == (1.0, 30.0)


def test_bench_cli_with_gpus_two_prints_one_line():
    """--gpus 2 without torch.distributed.run: bench.py starts the two ranks
    itself and rank 0 alone prints (the reference arm, which runs on CPU)."""
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                        "--warmup", "0", "--workload", "s64_b2_h384_bf16"], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    assert json.loads(lines[0])["n_gpus"] == 2
