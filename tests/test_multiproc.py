"""Multi-rank host logic on CPU (gloo, world size 2).

The path has no exchange step, so N GPUs run N independent replicas: each rank draws its
own inputs, times its own steps, and rank 0 reports the units all ranks processed divided
by the slowest rank's time.  These tests run that host logic on gloo without a GPU.
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


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    m = bench._max_over_ranks(float(rank + 1) * 3.0, ws, "cpu")
    s = bench._sum_over_ranks(10.0 * (rank + 1), ws, "cpu")
    seeds = [bench.replica_seed(1001, i, rank) for i in range(3)]
    q.put((rank, m, s, seeds))
    dist.destroy_process_group()


def test_replica_reductions_and_seeds_gloo():
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
    assert [r[1] for r in res] == [6.0, 6.0]           # max over ranks of per-rank times
    assert [r[2] for r in res] == [30.0, 30.0]         # sum over ranks of per-rank units
    s0, s1 = res[0][3], res[1][3]
    assert len(set(s0 + s1)) == 6                      # every replica and input set has its own seed


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["value"] > 0 and rec["unit"] == "GB/s"
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["e2e"]["h2d_bytes_per_step"] == 0
