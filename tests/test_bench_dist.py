"""bench.py's multi-process path on the CPU (gloo, world size 2): replicas, max over ranks,
and rank 0 alone printing the reference arm's line."""

import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r was slower on the first timing and faster on the second
        ms, vals = bench._aggregate_over_ranks(torch, world, [10.0 + 5 * rank, 8.0 - rank],
                                               [1000, 400], "cpu")
        out[rank] = (ms, vals)
    finally:
        dist.destroy_process_group()


def test_aggregate_takes_the_slowest_rank():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms, vals = res[rank]
        assert ms == [15.0, 8.0]
        assert vals == [world * 1000 / 15e-3, world * 400 / 8e-3]


def test_aggregate_single_process():
    ms, vals = bench._aggregate_over_ranks(torch, 1, [4.0], [100], "cpu")
    assert ms == [4.0] and vals == [100 / 4e-3]


def test_reference_arm_under_torchrun_prints_once():
    # two ranks on the host: rank 0 times the oracle and prints one JSON line, rank 1 exits 0
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["value"] > 0 and rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
