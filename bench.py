#!/usr/bin/env python3
"""Throughput of one GPT-2 training step (forward, backward, AdamW) on a B300.

Default workload: GPT-2 124M (V 50257, L 12, H 12, C 768) at B=16, T=1024 with
tensor-core contractions on bf16 operands (fp32 accumulation, fp32 master
weights; --mode tf32 or fp32 for the other arithmetic), seeded synthetic
parameters and a Zipf(1.1) token stream.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (single-precision build, OpenMP on the
host cores) on a bounded sample of the same workload.  Under torchrun every
rank runs an independent replica of the step (the path has no collective on
one GPU per rank); the timed region is bracketed by a barrier and the slowest
rank's time is used.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gpt_decoder_step_train_b300 import synthetic as syn  # noqa: E402

METRIC = "train tokens/s per fwd+bwd+AdamW step (GPT-2 124M, B16 T1024); % roofline"
UNIT = "tokens/s"
MEASURED_PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
# nominal dense tensor rates (PFLOP/s): tf32 1.1, bf16 2.25 -> ratio used to derive the
# tf32 peak from the measured bf16 peak
TF32_OVER_BF16 = 1.1 / 2.25


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="124M", choices=list(syn.CONFIGS))
    ap.add_argument("--mode", default="bf16", choices=["bf16", "tf32", "fp32"])
    ap.add_argument("--dropout", type=float, default=0.0,
                    help="dropout probability of the training step (default 0: the step without dropout)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-trace", action="store_true")
    ap.add_argument("--cpu-sample-T", type=int, default=256,
                    help="positions of the single sequence the CPU baseline runs")
    ap.add_argument("--op", default=None,
                    help="time one kernel of the workload in isolation (prints its own JSON line)")
    return ap.parse_args()


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ------------------------------------------------------------------ ranks
# One process per GPU, each running an independent replica of the step (the path
# has no data exchange on one GPU per rank).  These helpers take the device of the
# process group's backend: a CUDA device under NCCL, the CPU under gloo.
def barrier(world, cuda=True):
    """All ranks meet here; with cuda, the device is idle on both sides."""
    import torch
    if cuda:
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    if cuda:
        torch.cuda.synchronize()


def max_over_ranks(x, world, device):
    """The largest x over all ranks (the slowest rank's time)."""
    if world == 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, B, T, steps, ms_total):
    """Whole-job throughput: the tokens of every rank's timed steps over the
    slowest rank's time (weak scaling: B x T per rank)."""
    return world * B * T * steps / (ms_total / 1000.0)


def load_peaks():
    try:
        with open(MEASURED_PEAKS) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


def gemm_traffic_per_launch():
    """DRAM bytes per GEMM launch from the committed ncu summary, or None when the
    GEMM sources changed since it was taken (the summary records their hash)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "gemm_tc_124M_B16T1024_bf16_dram.md")
    try:
        fields = dict(line.split(": ", 1) for line in open(path).read().splitlines() if ": " in line
                      and line.split(": ", 1)[0] in ("traffic_bytes_per_launch", "sources", "sources_sha256"))
        h = hashlib.sha256()
        for f in fields["sources"].split():
            h.update(open(os.path.join(ROOT, f), "rb").read())
        if h.hexdigest() != fields["sources_sha256"].strip():
            return None
        return int(fields["traffic_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def gemm_flops(cfg, B, T):
    """Algorithmic FLOPs of every linear layer's forward, dX and dW product."""
    BT = B * T
    return 6.0 * BT * (12 * cfg.L * cfg.C ** 2 + cfg.C * cfg.V)


def step_flops(cfg, B, T):
    """Matmul FLOPs plus causal attention FLOPs (fwd + bwd) of one step."""
    return gemm_flops(cfg, B, T) + 6.0 * cfg.L * T * cfg.C * B * T


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for _, _, flags in rows for i, f in enumerate(flags)
                          if f.lower() == "active"})
        mx = max(r[1] for r in rows)
        loaded = [r[0] for r in rows if r[0] > 0.3 * mx] or [r[0] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------------ CPU oracle timing
def time_oracle(cfg, T_sample, steps, warmup=0):
    """Time the single-precision oracle on one sequence of T_sample positions of
    the workload (fwd + bwd + AdamW over all parameters).  Returns (tokens/s, cores)."""
    from oracle import Oracle
    o = Oracle("f32")
    params = syn.init_params(cfg)
    tok, tgt = syn.draw_tokens(cfg, B=1, T=T_sample)
    m = o.model(cfg.dims(), 1, T_sample)
    am, av = np.zeros_like(params), np.zeros_like(params)
    times = []
    for t in range(1, warmup + steps + 1):
        t0 = time.perf_counter()
        m.forward(params, tok, tgt)
        g = m.backward(params)
        m.adamw(params, g, am, av, cfg.lr, cfg.b1, cfg.b2, cfg.eps, cfg.wd, t)
        if t > warmup:
            times.append(time.perf_counter() - t0)
    return T_sample * len(times) / sum(times), o.num_threads(), sum(times)


# ------------------------------------------------------------------ reference arm
def run_reference(args, cfg):
    world, rank, _ = dist_info()
    if rank != 0:
        return 0
    T_sample = 64
    tps, cores, total = time_oracle(cfg, T_sample, args.steps, args.warmup)
    sample = (f"{args.steps} timed steps (+{args.warmup} warm-up), each fwd+bwd+AdamW of the "
              f"{cfg.name} model on one sequence of {T_sample} positions")
    line = {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * T_sample / tps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded init, Zipf(1.1) tokens)",
        "config": {"workload": cfg.name, "global_batch": cfg.B, "seq_len": cfg.T,
                   "sample": f"B=1 T={T_sample}", "parallelism": "cpu-openmp"},
        "cpu_baseline": {"value": tps, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": tps, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm
def run_ours(args, cfg):
    import torch
    from gpt_decoder_step_train_b300 import binding
    from gpt_decoder_step_train_b300.binding import GPT2

    world, rank, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    B, T = cfg.B, cfg.T

    params = torch.from_numpy(syn.init_params(cfg)).to(dev)
    model = GPT2(cfg, params, maxB=B, mode=args.mode)
    if args.dropout > 0:
        rc = model.set_dropout(args.dropout, 1234 + rank)
        if rc != 0:
            raise RuntimeError(f"set_dropout failed: {binding.strerror(rc)}")
    stream = model.stream
    # a pool of distinct batches (seeded per rank), resident on the device
    pool = []
    for i in range(4):
        tok, tgt = syn.draw_tokens(cfg, seed=cfg.token_seed + 1000 * rank + i)
        pool.append((tok, tgt))
    dev_pool = [(torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev)) for a, b in pool]
    host_pool = [(torch.from_numpy(a).pin_memory(), torch.from_numpy(b).pin_memory())
                 for a, b in pool]

    t_step = [0]

    def step(tokens, targets):
        t_step[0] += 1
        loss = model.forward(tokens, targets)
        rc = model.backward()
        if rc != 0:
            raise RuntimeError(f"backward failed: {binding.strerror(rc)}")
        rc = model.adamw(cfg.lr, cfg.b1, cfg.b2, cfg.eps, cfg.wd, t_step[0])
        if rc != 0:
            raise RuntimeError(f"adamw failed: {binding.strerror(rc)}")
        return loss

    for i in range(args.warmup):
        loss = step(*dev_pool[i % len(dev_pool)])
    st = model.status()
    if st != 0:
        raise RuntimeError(f"warm-up failed: {binding.strerror(st)}")

    # ---- timed region: inputs resident in HBM -------------------------------
    gpu_index = local
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    if vis:
        try:
            gpu_index = int(vis.split(",")[local])
        except ValueError:
            pass
    clocks = ClockSampler(gpu_index)
    barrier(world)
    clocks.start()
    n_launch0 = binding.lib().gpt2_kernel_launches()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    losses = []
    for i in range(args.steps):
        losses.append(step(*dev_pool[i % len(dev_pool)]))
    e1.record(stream)
    barrier(world)
    clock_info = clocks.stop()
    launches = binding.lib().gpt2_kernel_launches() - n_launch0
    ms_total = max_over_ranks(e0.elapsed_time(e1), world, dev)
    # per-kernel times: a second pass of the same steps with CUDA events around
    # every operation on the model's stream (kept out of the timed region above,
    # whose value the event records would slow by a few percent)
    kernels = {}
    if not args.no_trace:
        model.trace(True)
        barrier(world)
        for i in range(args.steps):
            step(*dev_pool[i % len(dev_pool)])
        barrier(world)
        kernels = model.trace_read()
        model.trace(False)
    st = model.status()
    if st != 0:
        raise RuntimeError(f"timed steps failed: {binding.strerror(st)}")
    if not all(np.isfinite(losses)):
        raise RuntimeError(f"non-finite loss: {losses}")

    ms_per_step = ms_total / args.steps
    value = job_tokens_per_s(world, B, T, args.steps, ms_total)

    # ---- end to end: pinned host inputs copied every step, loss read back ---
    e2e = None
    if not args.no_e2e:
        ke = max(3, min(args.steps, 10))
        barrier(world)
        t0 = time.perf_counter()
        for i in range(ke):
            step(*host_pool[i % len(host_pool)])
        barrier(world)
        wall = max_over_ranks(time.perf_counter() - t0, world, dev)
        e2e = {"value": world * B * T * ke / wall, "unit": UNIT,
               "h2d_bytes_per_step": 2 * B * T * 4, "d2h_bytes_per_step": 4, "steps": ke}

    # ---- roofline of the dominant kernel (the tcgen05 GEMM) ------------------
    peaks, peak_src = load_peaks()
    roofline = None
    per_class = {}
    if kernels:
        for name, (ms, nl) in kernels.items():
            per_class[name] = {"ms_per_step": round(ms / args.steps, 4),
                               "launches_per_step": nl / args.steps}
        gemm_names = ("matmul_fwd", "matmul_bwd_input", "matmul_bwd_weight")
        gemm_ms = sum(kernels[n][0] for n in gemm_names) / args.steps
        # the timed region is well under a second at full clocks: the burst peak
        # is the denominator; the sustained (power-capped) figure is given beside it
        ratio = {"tf32": TF32_OVER_BF16, "bf16": 1.0}.get(args.mode)
        if ratio is not None:
            peak = peaks["bf16_tflops"] * ratio
            peak_sus = peaks["bf16_tflops_sustained"] * ratio
            peak_note = (f"{args.mode} = bf16 burst x 1.1/2.25 (of {peak_src})" if args.mode == "tf32"
                         else f"bf16 burst (of {peak_src})")
        else:
            peak = peak_sus = None
            peak_note = "fp32 SIMT mode"
        achieved = gemm_flops(cfg, B, T) / (gemm_ms / 1000.0) / 1e12
        step_tf = step_flops(cfg, B, T) / (ms_per_step / 1000.0) / 1e12
        roofline = {"kernel": f"gemm_tc<{args.mode}> (all linear fwd/dX/dW products)", "bound": "tensor",
                    "achieved": round(achieved, 1), "peak": round(peak, 1) if peak else None,
                    "unit": "TFLOP/s", "frac": round(achieved / peak, 4) if peak else None,
                    "traffic": None, "peak_source": peak_note,
                    "frac_of_sustained": round(achieved / peak_sus, 4) if peak_sus else None,
                    "step_frac_of_burst": round(step_tf / peak, 4) if peak else None,
                    "share_of_step": round(gemm_ms / ms_per_step, 4)}
        if args.mode == "bf16" and args.config == "124M":
            # DRAM bytes per launch, from the committed ncu capture of this workload
            tr = gemm_traffic_per_launch()
            roofline["traffic"] = tr
            if tr is not None:
                roofline["traffic_unit"] = "bytes per launch (dram read + write, ncu)"

    mfu = step_flops(cfg, B, T) / (ms_per_step / 1000.0) / 1e12
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"tf32": "tf32", "bf16": "bf16", "fp32": "f32"}[args.mode],
        "data": "synthetic (seeded N(0,0.02) init, Zipf(1.1) tokens, next-token targets)",
        "config": {"workload": cfg.name, "global_batch": B * world, "seq_len": T,
                   "mode": args.mode, "parallelism": f"replicas{world}" if world > 1 else "single",
                   "dropout": args.dropout,
                   "l2": "working set ~15 GB >> 126 MB L2, no flush"},
        "loss_first_last": [round(losses[0], 5), round(losses[-1], 5)],
        "step_tflops": round(mfu, 1),
        "roofline": roofline,
        "kernels": per_class,
        "gpu_launches": int(launches),
        "clocks": clock_info,
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tps, cores, total = time_oracle(cfg, args.cpu_sample_T, 1)
        line["cpu_baseline"] = {
            "value": round(tps, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"one fwd+bwd+AdamW step of the same model on B=1, T={args.cpu_sample_T} "
                      f"(oracle, single-precision build), {total:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    model.close()
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


# ------------------------------------------------------------------ single-op timing
# name -> (description, builder); a builder returns (callable, algorithmic flops, bytes)
OPS = {}


def _op(name):
    def deco(f):
        OPS[name] = f
        return f
    return deco


def _gemm_case(kind, N, IC, OC, mode):
    import torch
    from gpt_decoder_step_train_b300 import binding as B_
    L = B_.lib()
    m = B_.MODES[mode]
    g = torch.Generator(device="cuda").manual_seed(0)
    x = torch.randn(N, IC, device="cuda", generator=g)
    w = torch.randn(OC, IC, device="cuda", generator=g) * 0.02
    dy = torch.randn(N, OC, device="cuda", generator=g)
    out = torch.empty(N, max(IC, OC), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    keep = [x, w, dy, out, st]
    if kind == "fwd":
        fn = lambda: L.gpt2_op_linear_forward(B_.ptr(out), None, B_.ptr(x), B_.ptr(w), None, None,
                                              N, IC, OC, OC, 0, m, B_.ptr(st), None)
    elif kind == "dx":
        fn = lambda: L.gpt2_op_linear_backward_input(B_.ptr(out), B_.ptr(dy), B_.ptr(w), None, N,
                                                     IC, OC, OC, m, B_.ptr(st), None)
    else:
        nbytes = L.gpt2_op_linear_backward_weight_scratch_bytes(N, IC, OC, m)
        sc = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        dw = torch.empty(OC, IC, device="cuda")
        keep += [sc, dw]
        fn = lambda: L.gpt2_op_linear_backward_weight(B_.ptr(dw), None, B_.ptr(dy), B_.ptr(x), N,
                                                      IC, OC, OC, B_.ptr(sc), nbytes, m,
                                                      B_.ptr(st), None)
    return fn, 2.0 * N * IC * OC, 4.0 * (N * IC + IC * OC + N * OC), keep


for _k in ("fwd", "dx", "dw"):
    for _nm, (_ic, _oc) in {"qkv": (768, 2304), "fc": (768, 3072), "fcproj": (3072, 768),
                           "attproj": (768, 768), "lmhead": (768, 50304)}.items():
        OPS[f"gemm_{_k}_{_nm}"] = (lambda k, ic, oc: (lambda mode: _gemm_case(k, 16384, ic, oc, mode)))(_k, _ic, _oc)


def _bgemm_case(name, M=16384, C=768, V=50257, Vp=50304):
    """One bf16 product of the step, with the epilogue the step gives it."""
    import ctypes as C_
    import torch
    from gpt_decoder_step_train_b300 import binding as B_
    L = B_.lib()
    g = torch.Generator(device="cuda").manual_seed(0)
    bf = torch.bfloat16

    def rnd(*shape, dtype=torch.float32, s=1.0):
        return (torch.randn(*shape, device="cuda", generator=g) * s).to(dtype)

    a = B_.gpt2_gemm_args()
    keep = []

    def put(field, t):
        keep.append(t)
        setattr(a, field, B_.ptr(t))
    kind, lay = name.split("_", 1)
    colsum = lay.endswith("cs")                        # with the per-32-row column sums (bias gradient)
    lay = lay[:-2] if colsum else lay
    dims = {"qkv": (C, 3 * C), "attproj": (C, C), "fc": (C, 4 * C), "fcproj": (4 * C, C), "lmhead": (C, V)}
    IC, OC = dims[lay]
    if kind == "fwd":                                  # out[M, OC] = x[M, IC] W[OC, IC]^T
        a.M, a.N, a.K = M, OC, IC
        put("A", rnd(M, IC, dtype=bf)); a.lda = IC; a.a_kmajor = 1
        put("B", rnd(OC, IC, dtype=bf, s=0.02)); a.ldb = IC; a.b_kmajor = 1
        ldo = Vp if lay == "lmhead" else OC
        if lay != "lmhead":
            put("bias", rnd(OC, s=0.02))
        if lay in ("attproj", "fcproj"):
            put("residual", rnd(M, ldo))
            put("out", rnd(M, ldo)); a.out_bf16 = 0
        elif lay == "fc":
            a.gelu = 1
            put("out_pre", rnd(M, ldo, dtype=bf)); a.pre_bf16 = 1
            put("out", rnd(M, ldo, dtype=bf)); a.out_bf16 = 1
        elif lay == "qkv":
            put("out", rnd(M, ldo, dtype=bf)); a.out_bf16 = 1
        else:
            put("out", torch.empty(M, ldo, device="cuda")); a.out_bf16 = 0
        a.ldo = ldo
    else:                                              # dx[M, IC] = dy[M, OC] W[OC, IC]
        a.M, a.N, a.K = M, IC, OC
        ldy = Vp if lay == "lmhead" else OC
        put("A", rnd(M, ldy, dtype=bf, s=0.01)); a.lda = ldy; a.a_kmajor = 1
        put("B", rnd(OC, IC, dtype=bf, s=0.02)); a.ldb = IC; a.b_kmajor = 0
        if lay == "fcproj":                            # dh = (dy W) * gelu'(h)
            put("gelu_x", rnd(M, IC, dtype=bf)); a.ldg = IC; a.gelu_x_bf16 = 1
            put("out", torch.empty(M, IC, device="cuda", dtype=bf)); a.out_bf16 = 1
        else:
            put("out", torch.empty(M, IC, device="cuda")); a.out_bf16 = 0
        a.ldo = IC
    if colsum:
        put("colsum", torch.empty((a.M + 31) // 32, a.N, device="cuda"))
    a.bf16 = 1
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    keep += [st, a]
    fn = lambda: L.gpt2_op_gemm(C_.byref(a), B_.MODES["bf16"], B_.ptr(st), None)
    return fn, 2.0 * a.M * a.N * a.K, 0.0, keep


for _k in ("fwd", "dx"):
    for _nm in ("qkv", "attproj", "fc", "fcproj", "lmhead"):
        OPS[f"bgemm_{_k}_{_nm}"] = (lambda n: (lambda mode: _bgemm_case(n)))(f"{_k}_{_nm}")
OPS["bgemm_dx_fcprojcs"] = lambda mode: _bgemm_case("dx_fcprojcs")


def _mem_case(name, N=16384, C=768, V=50257, Vp=50304):
    """One HBM-bound kernel of the step at its GPT-2 124M B16 T1024 size.  Returns
    the algorithmic bytes of one launch: every input read once, every output
    written once."""
    import torch
    from gpt_decoder_step_train_b300 import binding as B_
    L = B_.lib()
    g = torch.Generator(device="cuda").manual_seed(0)
    dev = "cuda"
    keep = []

    def k(t):
        keep.append(t)
        return B_.ptr(t)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    keep.append(st)
    if name == "ln_fwd":                               # x fp32 -> y bf16, mean, rstd
        x = torch.randn(N, C, device=dev, generator=g)
        w, b = torch.ones(C, device=dev), torch.zeros(C, device=dev)
        y = torch.empty(N, C, device=dev, dtype=torch.bfloat16)
        mu, rs = torch.empty(N, device=dev), torch.empty(N, device=dev)
        fn = lambda: L.gpt2_op_layernorm_forward_bf16(k(y), k(mu), k(rs), k(x), k(w), k(b), N, C, None)
        nbytes = N * C * (4 + 2) + 8 * N
    elif name == "ln_bwd":                             # dx += LN'(dy): dx fp32 (read+write) + bf16 copy
        x = torch.randn(N, C, device=dev, generator=g)
        dy = torch.randn(N, C, device=dev, generator=g)
        dx = torch.randn(N, C, device=dev, generator=g)
        dx16 = torch.empty(N, C, device=dev, dtype=torch.bfloat16)
        w = torch.ones(C, device=dev)
        mu, rs = torch.zeros(N, device=dev), torch.ones(N, device=dev)
        dw, db = torch.empty(C, device=dev), torch.empty(C, device=dev)
        nsc = L.gpt2_op_layernorm_backward_scratch_bytes(N, C)
        sc = torch.empty(nsc, dtype=torch.uint8, device=dev)
        ds = torch.empty(C, device=dev)
        fn = lambda: L.gpt2_op_layernorm_backward(k(dx), k(dx16), k(dw), k(db), k(ds), k(dy), k(x), k(w), k(mu),
                                                  k(rs), N, C, 1, k(sc), nsc, k(st), None)
        nbytes = N * C * (4 + 4 + 4 + 4 + 2) + 8 * N
    elif name == "crossentropy":                       # logits fp32 read, dlogits bf16 written
        z = torch.randn(N, Vp, device=dev, generator=g)
        dz = torch.empty(N, Vp, device=dev, dtype=torch.bfloat16)
        tgt = torch.randint(0, V, (N,), device=dev, dtype=torch.int32, generator=g)
        losses = torch.empty(N, device=dev)
        fn = lambda: L.gpt2_op_crossentropy(k(losses), k(z), k(dz), k(tgt), N, V, Vp, 1.0 / N, k(st), None)
        nbytes = N * V * (4 + 2) + 8 * N
    elif name == "crossentropy_bf16":                  # bf16 logits read, bf16 gradient written in place
        z = (torch.randn(N, Vp, device=dev, generator=g) * 2).to(torch.bfloat16)
        tgt = torch.randint(0, V, (N,), device=dev, dtype=torch.int32, generator=g)
        losses = torch.empty(N, device=dev)
        fn = lambda: L.gpt2_op_crossentropy_bf16(k(losses), k(z), k(tgt), N, V, Vp, 1.0 / N, k(st), None)
        nbytes = N * Vp * (2 + 2) + 8 * N
    elif name.startswith("bias_grad"):                 # column sums of dY [N, 3C] (bf16) or [N, C] (fp32)
        bf = name.endswith("bf16")
        OC = 3 * C if bf else C
        dout = torch.randn(N, OC, device=dev, generator=g).to(torch.bfloat16 if bf else torch.float32)
        db = torch.empty(OC, device=dev)
        nsc = L.gpt2_op_bias_grad_scratch_bytes(N, OC)
        sc = torch.empty(nsc, dtype=torch.uint8, device=dev)
        fn = lambda: L.gpt2_op_bias_grad(k(db), k(dout), int(bf), N, OC, OC, k(sc), nsc, None)
        nbytes = N * OC * (2 if bf else 4)
    elif name == "adamw":                              # p, g, m, v read; p, m, v written (124M params)
        n = 124439808
        p, gr = torch.randn(n, device=dev, generator=g), torch.randn(n, device=dev, generator=g)
        m_, v_ = torch.zeros(n, device=dev), torch.zeros(n, device=dev)
        fn = lambda: L.gpt2_op_adamw(k(p), k(gr), k(m_), k(v_), n, 1e-4, 0.9, 0.999, 1e-8, 0.0, 0.1, 0.001, None)
        nbytes = 28 * n
    elif name == "encoder_fwd":                        # token and position rows gathered, x written
        B_n, T = 16, 1024
        wte = torch.randn(V, C, device=dev, generator=g)
        wpe = torch.randn(1024, C, device=dev, generator=g)
        tok = torch.randint(0, V, (B_n, T), device=dev, dtype=torch.int32, generator=g)
        x = torch.empty(B_n * T, C, device=dev)
        fn = lambda: L.gpt2_op_encoder_forward(k(x), k(tok), k(wte), k(wpe), B_n, T, C, V, k(st), None)
        nbytes = B_n * T * C * 4 * 3
    else:
        raise KeyError(name)
    return fn, 0.0, float(nbytes), keep


for _nm in ("ln_fwd", "ln_bwd", "crossentropy", "crossentropy_bf16", "bias_grad_bf16", "bias_grad_f32", "adamw", "encoder_fwd"):
    OPS[f"mem_{_nm}"] = (lambda n: (lambda mode: _mem_case(n)))(_nm)


def _attn_case(kind, mode, B=16, T=1024, C=768, H=12):
    import torch
    from gpt_decoder_step_train_b300 import binding as B_
    L = B_.lib()
    m = B_.MODES[mode]
    dt = torch.bfloat16 if mode == "bf16" else torch.float32
    g = torch.Generator(device="cuda").manual_seed(0)
    qkv = torch.randn(B, T, 3 * C, device="cuda", generator=g).to(dt)
    y = torch.empty(B, T, C, device="cuda", dtype=dt)
    lse = torch.empty(B, H, T, device="cuda")
    dy = torch.randn(B, T, C, device="cuda", generator=g).to(dt)
    dqkv = torch.empty_like(qkv)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    nbytes = L.gpt2_op_attention_backward_scratch_bytes(B, T, H)
    sc = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    keep = [qkv, y, lse, dy, dqkv, st, sc]
    L.gpt2_op_attention_forward(B_.ptr(y), B_.ptr(lse), B_.ptr(qkv), B, T, C, H, m, B_.ptr(st), None)
    causal_pairs = B * H * T * (T + 1) / 2
    hs = C // H
    if kind == "fwd":
        fn = lambda: L.gpt2_op_attention_forward(B_.ptr(y), B_.ptr(lse), B_.ptr(qkv), B, T, C, H, m,
                                                 B_.ptr(st), None)
        flops = 4.0 * hs * causal_pairs
    else:
        fn = lambda: L.gpt2_op_attention_backward(B_.ptr(dqkv), B_.ptr(dy), B_.ptr(qkv), B_.ptr(y),
                                                  B_.ptr(lse), B, T, C, H, B_.ptr(sc), nbytes, m,
                                                  B_.ptr(st), None)
        flops = 8.0 * hs * causal_pairs
    return fn, flops, qkv.element_size() * (qkv.numel() + 2 * y.numel()), keep


OPS["attn_fwd"] = lambda mode: _attn_case("fwd", mode)
OPS["attn_bwd"] = lambda mode: _attn_case("bwd", mode)


def _decode_case(mode, B=1, steps=64):
    """Autoregressive decoding with the key/value cache: one call decodes positions
    0 .. steps-1 of B rows (GPT-2 124M); every step reads each fp32 weight once."""
    import numpy as np
    import torch
    from gpt_decoder_step_train_b300 import synthetic as syn
    from gpt_decoder_step_train_b300.binding import GPT2
    cfg = syn.CONFIGS["124M"]
    params = torch.from_numpy(syn.init_params(cfg)).cuda()
    model = GPT2(cfg, params, maxB=B, mode=mode)
    tok = torch.from_numpy(np.asarray(syn.draw_tokens(cfg)[0][:B, :steps], dtype=np.int32)).cuda()
    cols = [tok[:, t].contiguous() for t in range(steps)]
    out = torch.empty(B, cfg.V, device="cuda")

    def fn():
        rc = 0
        for t in range(steps):
            rc = rc or model.decode(cols[t], t, out)
        return rc
    n = syn.num_params(cfg)
    return fn, 2.0 * n * B * steps, 4.0 * n * steps, [model, params, tok, cols, out]


OPS["decode"] = _decode_case


def run_op(args):
    """Time single operations: --op takes names or prefixes, comma separated."""
    import torch
    torch.cuda.set_device(0)
    names = [n for want in args.op.split(",") for n in sorted(OPS) if n == want or n.startswith(want)]
    if not names:
        print(f"unknown op {args.op!r}; known: {', '.join(sorted(OPS))}", file=sys.stderr)
        return 2
    peaks, src = load_peaks()
    for name in names:
        fn, flops, nbytes, keep = OPS[name](args.mode)
        for _ in range(args.warmup):
            assert fn() == 0
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            assert fn() == 0
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        bf16 = args.mode == "bf16" or name.startswith("bgemm")
        peak = peaks["bf16_tflops"] * (1.0 if bf16 else TF32_OVER_BF16)
        tf = flops / (ms / 1e3) / 1e12
        gbs = nbytes / (ms / 1e3) / 1e9 if nbytes else None
        print(json.dumps({"op": name, "mode": "bf16" if bf16 else args.mode, "ms": round(ms, 4),
                          "tflops": round(tf, 1) if flops else None,
                          "frac_of_burst_peak": round(tf / peak, 3) if flops else None,
                          "gbs_algorithmic": round(gbs, 1) if gbs else None,
                          "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 3) if gbs else None}),
              flush=True)
        del keep
    return 0


def main():
    args = parse_args()
    if args.op:
        return run_op(args)
    cfg = syn.CONFIGS[args.config]
    if args.impl == "reference":
        return run_reference(args, cfg)
    return run_ours(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
