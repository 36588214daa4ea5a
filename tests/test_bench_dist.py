"""Multi-rank host logic of bench.py on CPU with the gloo backend (world size 2).

The bench runs one replica per rank; what is shared across ranks is the
timing protocol: a barrier on both sides of the timed region, the slowest
rank's time, and the whole-job throughput.  These run here without a GPU.
"""
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


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.rank_barrier()
    slowest = bench.reduce_max(1.5 + rank, "cpu")   # rank r "took" 1.5 + r ms
    value = bench.whole_job_tflops(world, 2.0e12, slowest)
    bench.rank_barrier()
    out[rank] = (slowest, value)
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_throughput():
    world = 2
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1]
    slowest, value = out[0]
    assert slowest == 2.5
    assert abs(value - world * 2.0e12 / 2.5e-3 / 1e12) < 1e-9


def test_single_process_helpers():
    import bench
    assert bench.reduce_max(3.25, "cpu") == 3.25
    assert bench.whole_job_tflops(1, 1e12, 1.0) == 1000.0


def test_reference_arm_prints_one_line_under_torchrun():
    """--impl reference under two ranks: rank 0 prints the line, rank 1 exits 0."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--ref-tokens", "128"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
