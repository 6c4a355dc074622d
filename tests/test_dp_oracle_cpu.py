"""Data parallelism's one exchange step, checked with the oracle on two CPU
ranks over gloo (127.0.0.1): each rank runs forward and backward on its half of
the batch, the ranks average their gradients with an all-reduce (sum / 2) and
apply the same AdamW step; the result equals one full-batch step.  The mean
loss over B*T positions is the mean of the two half-batch means when the halves
have equal size, so the averaged gradient is the full-batch gradient.

A rank that fails before the exchange is seen by the other on the host: its
all-reduce raises within the process group's timeout instead of waiting
forever.  No GPU is used here."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

from gpt_decoder_step_train_b300 import synthetic as syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


_RANK_CODE = r"""
import datetime, json, os, sys
sys.path.insert(0, os.environ["DP_ROOT"])
import numpy as np
import torch
import torch.distributed as dist
from gpt_decoder_step_train_b300 import synthetic as syn
from oracle import Oracle

rank, world = int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"])
fail = os.environ.get("DP_FAIL_RANK") == str(rank)
dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=10))
cfg = syn.CONFIGS["tiny"]
o = Oracle("f64")
params = syn.init_params(cfg).astype(np.float64)
tok, tgt = syn.draw_tokens(cfg)
half = cfg.B // world
rows = slice(rank * half, (rank + 1) * half)
m = o.model(cfg.dims(), half, cfg.T)
am, av = np.zeros_like(params), np.zeros_like(params)
loss = m.forward(params, tok[rows], tgt[rows])
g = m.backward(params)
if fail:
    os._exit(3)                        # this rank dies before the exchange
t = torch.from_numpy(g)
try:
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    lt = torch.tensor([loss], dtype=torch.float64)
    dist.all_reduce(lt, op=dist.ReduceOp.SUM)
except Exception as e:                 # the peer is gone: reported, not waited for
    print(json.dumps({"rank": rank, "peer_failed": type(e).__name__}), flush=True)
    os._exit(0)
g = (t / world).numpy()
m.adamw(params, g, am, av, cfg.lr, cfg.b1, cfg.b2, cfg.eps, 0.1, 1)
np.save(os.path.join(os.environ["DP_OUT"], f"rank{rank}.npy"), np.concatenate([g, params]))
print(json.dumps({"rank": rank, "loss": float(lt.item()) / world}), flush=True)
dist.destroy_process_group()
"""


def _launch(tmp_path, fail_rank=None):
    from oracle import Oracle
    Oracle("f64")                      # build the oracle once, before the ranks start
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                   WORLD_SIZE="2", DP_ROOT=ROOT, DP_OUT=str(tmp_path), CUDA_VISIBLE_DEVICES="",
                   OMP_NUM_THREADS="2")
        if fail_rank is not None:
            env["DP_FAIL_RANK"] = str(fail_rank)
        procs.append(subprocess.Popen([sys.executable, "-c", _RANK_CODE], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    results = []
    for p in procs:
        out, err = p.communicate(timeout=180)
        lines = [l for l in out.splitlines() if l.startswith("{")]
        results.append((p.returncode, json.loads(lines[-1]) if lines else None, err))
    return results


def test_two_ranks_with_averaged_gradients_equal_one_full_batch_step(o64, tmp_path):
    res = _launch(tmp_path)
    for rc, msg, err in res:
        assert rc == 0, err[-2000:]
    cfg = syn.CONFIGS["tiny"]
    params = syn.init_params(cfg).astype(np.float64)
    tok, tgt = syn.draw_tokens(cfg)
    m = o64.model(cfg.dims(), cfg.B, cfg.T)
    loss = m.forward(params, tok, tgt)
    g = m.backward(params)
    p = params.copy()
    am, av = np.zeros_like(p), np.zeros_like(p)
    m.adamw(p, g, am, av, cfg.lr, cfg.b1, cfg.b2, cfg.eps, 0.1, 1)
    n = params.size
    r0, r1 = (np.load(tmp_path / f"rank{r}.npy") for r in range(2))
    assert np.array_equal(r0, r1)                      # both replicas hold the same state
    scale = np.abs(g).max()
    assert np.abs(r0[:n] - g).max() <= 1e-12 * scale  # averaged half-batch gradients
    assert np.abs(r0[n:] - p).max() <= 1e-12           # the same update as one full step
    for _, msg, _ in res:
        assert abs(msg["loss"] - loss) <= 1e-12


def test_a_rank_that_dies_before_the_exchange_is_reported_not_waited_for(tmp_path):
    res = _launch(tmp_path, fail_rank=1)
    (rc0, msg0, err0), (rc1, _, _) = res
    assert rc1 == 3
    assert rc0 == 0, err0[-2000:]
    assert msg0 is not None and "peer_failed" in msg0, msg0
