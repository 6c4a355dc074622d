"""Seeded synthetic inputs: model configurations, initial parameters, token batches.

This module holds no arithmetic of the training step.  It only draws the
inputs that both the CUDA path and the CPU oracle consume, so both see the
same bytes.

Inputs stand in for the pages' workloads (pretrained GPT-2 weights fine-tuned
on tinyshakespeare, and a 65-character vocabulary for the tiny model), which
are not available offline:
  * parameters: N(0, 0.02) for the embeddings and the fc / qkv weights,
    N(0, 0.02/sqrt(2L)) for the two residual projections (attention c_proj and
    MLP c_proj), biases 0, LayerNorm gain 1 and shift 0.  Drawn with NumPy's
    PCG64 from a stated seed, float32.
  * tokens: i.i.d. uniform over [0, V) for the tiny model; a truncated Zipf law
    P(id = k) proportional to (k+1)^-1.1 over [0, V) for the GPT-2 vocabularies,
    drawn by inverse CDF.  Each row draws T+1 tokens; inputs are the first T,
    targets the last T (next-token prediction).
"""
from dataclasses import dataclass, field

import numpy as np

TENSOR_NAMES = ("wte", "wpe", "ln1w", "ln1b", "qkvw", "qkvb", "attprojw", "attprojb",
                "ln2w", "ln2b", "fcw", "fcb", "fcprojw", "fcprojb", "lnfw", "lnfb")


@dataclass(frozen=True)
class Config:
    name: str
    V: int
    maxT: int
    L: int
    H: int
    C: int
    B: int
    T: int
    lr: float
    wd: float
    b1: float = 0.9
    b2: float = 0.999
    eps: float = 1e-8
    tokens: str = "zipf"          # "uniform" or "zipf"
    zipf_s: float = 1.1
    param_seed: int = 0
    token_seed: int = 1
    extra: dict = field(default_factory=dict, compare=False)

    def dims(self):
        return dict(V=self.V, maxT=self.maxT, L=self.L, H=self.H, C=self.C)

    def with_(self, **kw):
        d = {k: getattr(self, k) for k in self.__dataclass_fields__}
        d.update(kw)
        return Config(**d)


CONFIGS = {
    "tiny": Config("gpt2-tiny-V65-B4T32", V=65, maxT=64, L=2, H=4, C=64, B=4, T=32,
                   lr=1e-4, wd=0.0, tokens="uniform"),
    "124M_small": Config("gpt2-124M-B4T64", V=50257, maxT=1024, L=12, H=12, C=768, B=4, T=64,
                         lr=1e-4, wd=0.0),
    "124M": Config("gpt2-124M-B16T1024", V=50257, maxT=1024, L=12, H=12, C=768, B=16,
                   T=1024, lr=6e-4, wd=0.1),
    "350M": Config("gpt2-350M-B8T1024", V=50257, maxT=1024, L=24, H=16, C=1024, B=8,
                   T=1024, lr=6e-4, wd=0.1),
    "1.5B": Config("gpt2-1.5B-B4T1024", V=50257, maxT=1024, L=48, H=25, C=1600, B=4,
                   T=1024, lr=6e-4, wd=0.1),
}


def tensor_shapes(cfg):
    V, maxT, L, C = cfg.V, cfg.maxT, cfg.L, cfg.C
    return {
        "wte": (V, C), "wpe": (maxT, C),
        "ln1w": (L, C), "ln1b": (L, C),
        "qkvw": (L, 3 * C, C), "qkvb": (L, 3 * C),
        "attprojw": (L, C, C), "attprojb": (L, C),
        "ln2w": (L, C), "ln2b": (L, C),
        "fcw": (L, 4 * C, C), "fcb": (L, 4 * C),
        "fcprojw": (L, C, 4 * C), "fcprojb": (L, C),
        "lnfw": (C,), "lnfb": (C,),
    }


def num_params(cfg):
    return int(sum(int(np.prod(s)) for s in tensor_shapes(cfg).values()))


def tensor_offsets(cfg):
    """name -> (offset, size) in the flat parameter array."""
    out, off = {}, 0
    for name in TENSOR_NAMES:
        n = int(np.prod(tensor_shapes(cfg)[name]))
        out[name] = (off, n)
        off += n
    return out


ZERO_INIT = ("ln1b", "qkvb", "attprojb", "ln2b", "fcb", "fcprojb", "lnfb")


def init_params(cfg, seed=None, perturbed=False):
    """Flat float32 parameter array in the 16-tensor layout.

    perturbed=True additionally draws the biases and LayerNorm shifts from
    N(0, 0.02) and the LayerNorm gains from 1 + N(0, 0.02), so no tensor starts
    at an exact constant (a parameter state reached after some training)."""
    rng = np.random.Generator(np.random.PCG64(cfg.param_seed if seed is None else seed))
    shapes = tensor_shapes(cfg)
    out = np.empty(num_params(cfg), dtype=np.float32)
    resid_std = 0.02 / np.sqrt(2.0 * cfg.L)
    for name, (off, n) in tensor_offsets(cfg).items():
        seg = out[off:off + n]
        if name in ("wte", "wpe", "qkvw", "fcw"):
            seg[:] = rng.standard_normal(n, dtype=np.float32) * np.float32(0.02)
        elif name in ("attprojw", "fcprojw"):
            seg[:] = rng.standard_normal(n, dtype=np.float32) * np.float32(resid_std)
        elif name in ("ln1w", "ln2w", "lnfw"):
            seg[:] = 1.0
            if perturbed:
                seg += rng.standard_normal(n, dtype=np.float32) * np.float32(0.02)
        else:
            seg[:] = 0.0
            if perturbed:
                seg[:] = rng.standard_normal(n, dtype=np.float32) * np.float32(0.02)
        assert seg.size == int(np.prod(shapes[name]))
    return out


def zipf_cdf(V, s):
    w = np.arange(1, V + 1, dtype=np.float64) ** (-s)
    c = np.cumsum(w)
    return c / c[-1]


def draw_tokens(cfg, B=None, T=None, seed=None):
    """(inputs, targets), both int32 [B, T]; targets are inputs shifted by one."""
    B = cfg.B if B is None else B
    T = cfg.T if T is None else T
    rng = np.random.Generator(np.random.PCG64(cfg.token_seed if seed is None else seed))
    if cfg.tokens == "uniform":
        seq = rng.integers(0, cfg.V, size=(B, T + 1), dtype=np.int64)
    else:
        cdf = zipf_cdf(cfg.V, cfg.zipf_s)
        u = rng.random(size=(B, T + 1))
        seq = np.minimum(np.searchsorted(cdf, u, side="right"), cfg.V - 1)
    seq = seq.astype(np.int32)
    return np.ascontiguousarray(seq[:, :T]), np.ascontiguousarray(seq[:, 1:])
