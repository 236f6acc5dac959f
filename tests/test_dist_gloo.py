"""The multi-rank host logic of bench.py on CPU (gloo, world size 2).

Rows of the path are independent, so N GPUs run N replicas with no
data-path collective; the only cross-rank steps are the barrier around the
timed region and the maximum of the per-rank times.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, lr = bench.dist_env()
    assert (w, r, lr) == (world, rank, rank)
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    t = 1.0 + rank * 0.5               # per-rank "elapsed time"
    q.put((rank, bench.max_over_ranks(t, w)))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=5) for _ in range(2))
    assert got == {0: 1.5, 1: 1.5}


def test_single_rank_defaults(monkeypatch):
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.max_over_ranks(2.5, 1) == 2.5


def test_reference_arm_line_shape():
    # --impl reference times the oracle on a bounded sample; check its JSON line
    import argparse
    import bench
    args = argparse.Namespace(steps=1, warmup=0, workload="cfg1")
    line = bench.run_reference(args, ["cfg1"], 1, 0)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "impl", "cpu_baseline", "e2e", "config"):
        assert key in line
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
