"""bench.py's multi-rank logic on the CPU: two gloo ranks (one process each).

The GPU arm runs one replica per rank (the (b, h) problems are independent:
weak scaling, no data-path collective); its timing takes the slowest rank
and its value counts every rank's tokens. These are host functions, checked
here with gloo; the reference arm is run under torchrun with two ranks."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        barrier, max_over_ranks = bench.dist_helpers(world, "cpu")
        barrier()
        slowest = max_over_ranks(1.5 + rank)          # rank r "took" 1.5 + r seconds
        q.put((rank, slowest, bench.job_throughput(world, 100, slowest)))
        barrier()
    finally:
        dist.destroy_process_group()


def test_dist_helpers_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    # both ranks see the slowest rank's time; the job counts both ranks' units
    assert [r[1] for r in res] == [2.5, 2.5]
    assert all(abs(r[2] - 2 * 100 / 2.5) < 1e-12 for r in res)


def test_single_rank_helpers_are_plain():
    sys.path.insert(0, ROOT)
    import bench
    barrier, max_over_ranks = bench.dist_helpers(1, "cpu")
    assert barrier() is None and max_over_ranks(3.25) == 3.25
    assert bench.job_throughput(1, 1000, 0.5) == 2000


def test_reference_arm_under_torchrun_two_ranks():
    """Rank 0 alone times the oracle and prints one JSON line; rank 1 exits 0."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--ref-budget", "0.05"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["value"] == d["value"]
