"""The multi-GPU path is replicas only (no collective on the data path): each rank runs
the whole workload on its own GPU, the job's step time is the slowest rank's and the
whole-job value counts every rank's bytes.  These tests drive that host logic with
world-size-2 gloo process groups on CPU, and the reference arm under torchrun."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from tests._helpers import ROOT


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        us = 10.0 + 5.0 * rank                 # rank 1 is the slower replica
        m = bench._max_over_ranks(us, torch.device("cpu"))
        q.put((rank, m, bench._job_value(world, 2.0e9, m)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_and_count_every_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    assert [g[1] for g in got] == [15.0, 15.0]
    assert got[0][2] == pytest.approx(2 * 2.0e9 / 15.0e-6 / 1e9)


def test_single_process_keeps_its_own_time():
    assert bench._max_over_ranks(12.5, torch.device("cpu")) == 12.5
    assert bench._job_value(1, 1.0e9, 1.0e6) == pytest.approx(1.0)


def test_reference_arm_under_torchrun_prints_once():
    """Rank 0 alone times the oracle and prints one JSON line; rank 1 exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0", "--cpu-seconds", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["value"] > 0
    assert res["cpu_baseline"]["kind"] == "oracle" and res["e2e"]["h2d_bytes_per_step"] == 0
