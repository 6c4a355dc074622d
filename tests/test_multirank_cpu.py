"""The N > 1 launch path of bench.py, on CPU ranks over gloo (127.0.0.1).

The step has no data exchange when each rank owns one GPU: every rank runs an
independent replica, the ranks meet at a barrier around the timed region, and
the slowest rank's time gives the whole-job throughput (tokens of all ranks).
Under torchrun the reference arm (the CPU oracle) runs on rank 0 alone; the
other ranks exit 0 without work.  No GPU is used here."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


_RANK_CODE = r"""
import json, os, sys
sys.path.insert(0, os.environ["BENCH_ROOT"])
import torch.distributed as dist
import bench
world, rank, _ = bench.dist_info()
dist.init_process_group("gloo", rank=rank, world_size=world)
ms = [3.0, 5.0][rank]                  # this rank's timed milliseconds
bench.barrier(world, cuda=False)
slowest = bench.max_over_ranks(ms, world, "cpu")
value = bench.job_tokens_per_s(world, 16, 1024, 20, slowest)
bench.barrier(world, cuda=False)
dist.destroy_process_group()
print(json.dumps({"rank": rank, "slowest": slowest, "value": value}))
"""


def test_two_ranks_take_the_slowest_time_and_count_every_ranks_tokens():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                   LOCAL_RANK=str(rank), WORLD_SIZE="2", BENCH_ROOT=ROOT, CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", _RANK_CODE], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=240)
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for o in outs:
        assert o["slowest"] == 5.0
        assert o["value"] == pytest.approx(2 * 16 * 1024 * 20 / 0.005)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5, 1, "cpu") == 7.5
    assert bench.job_tokens_per_s(1, 4, 32, 10, 1000.0) == 4 * 32 * 10


def test_reference_arm_under_torchrun_prints_once_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--config", "tiny", "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
