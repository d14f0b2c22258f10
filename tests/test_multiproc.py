"""Multi-process plumbing on CPU (gloo, world size 2).

The path shards by request with no exchange: every rank runs its own replica
batch and only the timing is reduced (max over ranks). These tests run that
plumbing with the gloo backend, no GPU.
"""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_cache_42_gb300 import workloads as wl
    r, ws, local, dist = bench.dist_setup()
    assert (r, ws) == (rank, world) and dist.get_backend() == "gloo"
    # each rank times something different; every rank must see the max
    got = bench.max_over_ranks(float(10 * (rank + 1)), dist)
    # replica batches: same shape, different content per rank
    w = wl.make_config(1, seed=42 + 1 + 1000 * rank)
    q.put((rank, got, int(w.q.astype(np.int64).sum()), w.q.shape))
    bench.barrier(dist)
    dist.destroy_process_group()


def test_max_over_ranks_and_replica_batches():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [20.0, 20.0]
    assert res[0][3] == res[1][3] and res[0][2] != res[1][2]


@pytest.mark.slow
def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--config", "1", "--steps", "3", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
