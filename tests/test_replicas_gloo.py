"""The multi-replica path of bench.py on CPU: two gloo ranks (world size 2).

Tokens are independent, so N GPUs run N replicas with no data-path
collective; the only collective is the max over ranks of the timed seconds.
These tests run that aggregation and the reference arm's rank handling in two
processes on the host (no GPU)."""
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


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        seconds = [0.5, 2.0][rank]                     # rank 1 is the slow replica
        slowest = bench.max_over_ranks(seconds, ws)
        tput = bench.replica_throughput(100, seconds, ws)
        dist.barrier()
        q.put((rank, slowest, tput))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_throughput_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, slowest, tput in got:
        assert slowest == 2.0                          # both ranks see the slowest replica's time
        assert tput == pytest.approx(200 / 2.0)        # 2 replicas x 100 tokens over 2 s


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.replica_throughput(64, 2.0, 1) == 32.0


def test_reference_arm_under_torchrun_prints_only_on_rank0():
    """`bench.py --impl reference` launched as two ranks: rank 0 times the oracle
    and prints one JSON line, rank 1 exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--config", "1", "--steps", "1", "--warmup", "1"]
    env = dict(os.environ, OPENBLAS_NUM_THREADS="2", OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    import json
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
