"""The N > 1 path of bench.py on the CPU: ranks as gloo processes (world size 2).

The decode shards into independent replicas (each rank its own seeded workload, no
collective on the data path); the only exchange is the max over ranks of the timed
region, so a slow rank sets the job's time.  The reference arm (the oracle on the host
cores) runs on rank 0 alone under torchrun; the other ranks exit 0 without work.
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
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _max_worker(rank: int, ws: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        # every rank times a different step; each must report the slowest
        got = bench.max_over_ranks(10.0 + 5.0 * rank, ws, torch.device("cpu"))
        q.put((rank, got))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_max_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert res == [(0, 15.0), (1, 15.0)]


def test_max_over_ranks_single_rank_is_identity():
    assert bench.max_over_ranks(3.25, 1, torch.device("cpu")) == 3.25


def test_ranks_draw_independent_workloads():
    """Each rank's replica has its own seed (bench: seed + 1000 * rank): same shapes,
    different values, so no two ranks time the same data."""
    cfg = W.get("tiny")
    w0 = W.make_workload(cfg, seed=cfg.seed)
    w1 = W.make_workload(cfg, seed=cfg.seed + 1000)
    assert w0.q.shape == w1.q.shape and w0.k_cache.shape == w1.k_cache.shape
    assert not torch.equal(w0.q, w1.q)
    assert torch.equal(w0.context_lens, w1.context_lens)  # explicit lengths of the tiny workload


@pytest.mark.timeout(600)
def test_reference_arm_under_torchrun_two_ranks():
    """`bench.py --impl reference` launched as the driver launches it for N = 2: rank 0
    prints one JSON line, rank 1 prints nothing, both exit 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--config", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env={**os.environ, "OMP_NUM_THREADS": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
