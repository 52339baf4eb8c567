"""The bench's multi-rank logic on CPU with two gloo ranks: the slowest rank's time is taken,
and whole-job throughput counts every rank's work (weak scaling: independent (batch, head)
problems per rank, no collective on the data path).  Also runs the reference arm under a
two-rank launch: rank 0 alone prints, the other rank exits 0 without work."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 2.0 + rank  # rank 1 is the slower one
    slowest = bench.max_over_ranks(ms, world)
    tflops = bench.job_tflops(1e12, world, slowest)
    out[rank] = (slowest, tflops)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        slowest, tflops = out[r]
        assert slowest == 3.0
        assert tflops == pytest.approx(world * 1e12 / 3e-3 / 1e12)


def test_reference_arm_under_two_ranks_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--workload", "b1h1n256d64_bf16", "--steps", "1",
           "--warmup", "3", "--ref-step-s", "0.2"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
