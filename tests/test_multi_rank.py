"""Multi-process host logic of the benchmark, on CPU with the gloo backend.

The dense GEMV does not shard under the problem's scope (one GPU, no
collectives), so `bench.py --gpus N` runs N independent replicas: each rank
times its own workload, the timed region is the slowest rank's, `value` sums
every rank's bytes, and only rank 0 prints.  These tests run that logic with
two gloo ranks (no GPU), and the CPU reference arm under a two-rank launch.
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


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    elapsed = 0.25 if rank == 0 else 0.5  # the slower rank sets the timed region
    out = bench.replica_aggregate(torch, dist, world, elapsed, 1000, 10)
    dist.barrier()
    q.put((rank, out))
    dist.destroy_process_group()


def test_replica_aggregate_takes_max_over_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in range(world):
        elapsed, per_step, value = res[rank]
        assert elapsed == 0.5 and per_step == 0.05
        assert value == pytest.approx(2 * 1000 * 10 / 0.5 / 1e9)


def test_single_rank_aggregate_needs_no_process_group():
    import bench
    assert bench.replica_aggregate(torch, None, 1, 2.0, 500, 4) == (2.0, 0.5, 1e-6)


def test_reference_arm_under_two_ranks_prints_once():
    # torchrun with two CPU ranks: rank 0 times the oracle and prints one JSON
    # line; rank 1 exits 0 without output
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
