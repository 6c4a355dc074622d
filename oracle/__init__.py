"""NumPy bindings for the plain-C CPU oracle of one GPT-2 training step.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use this package; the product library never does.

``Oracle("f64")`` is the double-precision build (the parity reference);
``Oracle("f32")`` is the single-precision build (timed as the CPU baseline).
Arrays are NumPy, C-contiguous, of the build's dtype; token arrays are int32.
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

NTENSORS = 16
TENSOR_NAMES = ("wte", "wpe", "ln1w", "ln1b", "qkvw", "qkvb", "attprojw", "attprojb",
                "ln2w", "ln2b", "fcw", "fcb", "fcprojw", "fcprojb", "lnfw", "lnfb")
# activations exposed by oracle_act(which, layer)
ACT = {"x0": 0, "ln1": 1, "qkv": 2, "atty": 3, "res2": 4, "ln2": 5, "h": 6, "g": 7,
       "res3": 8, "lnf": 9, "P": 10, "ln1_mean": 11, "ln1_rstd": 12}

_libs = {}


def _load(precision):
    if precision in _libs:
        return _libs[precision]
    path = _build.lib_path(precision)
    if not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_build.SRC):
        _build.build()
    lib = C.CDLL(path)
    _libs[precision] = lib
    return lib


def _ptr(a):
    return a.ctypes.data_as(C.c_void_p) if a is not None else None


class Oracle:
    """Thin wrapper over one oracle build."""

    def __init__(self, precision="f64"):
        assert precision in ("f64", "f32")
        self.precision = precision
        self.lib = _load(precision)
        self.dtype = np.float64 if precision == "f64" else np.float32
        self.ctreal = C.c_double if precision == "f64" else C.c_float
        L = self.lib
        vp, i, sz = C.c_void_p, C.c_int, C.c_size_t
        r = self.ctreal
        L.oracle_real_bytes.restype = i
        assert L.oracle_real_bytes() == np.dtype(self.dtype).itemsize
        L.oracle_num_threads.restype = i
        L.oracle_num_params.restype = sz
        L.oracle_num_params.argtypes = [i, i, i, i]
        L.oracle_param_sizes.argtypes = [i, i, i, i, vp]
        L.oracle_encoder_forward.argtypes = [vp, vp, vp, vp, i, i, i]
        L.oracle_encoder_backward.argtypes = [vp, vp, vp, vp, i, i, i]
        L.oracle_layernorm_forward.argtypes = [vp, vp, vp, vp, vp, vp, i, i]
        L.oracle_layernorm_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i]
        L.oracle_matmul_forward.argtypes = [vp, vp, vp, vp, i, i, i]
        L.oracle_matmul_backward.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i]
        L.oracle_attention_forward.argtypes = [vp, vp, vp, i, i, i, i]
        L.oracle_attention_backward.argtypes = [vp, vp, vp, vp, i, i, i, i]
        L.oracle_attention_forward_dropout.argtypes = [vp, vp, vp, i, i, i, i, vp, C.c_double]
        L.oracle_attention_backward_dropout.argtypes = [vp, vp, vp, vp, i, i, i, i, vp, C.c_double]
        L.oracle_philox4x32_10.argtypes = [vp, vp, vp]
        L.oracle_dropout_keep.argtypes = [vp, sz, C.c_uint64, C.c_uint32, C.c_uint32, C.c_double]
        L.oracle_dropout_apply.argtypes = [vp, vp, vp, sz, C.c_double]
        L.oracle_set_dropout.restype = i
        L.oracle_set_dropout.argtypes = [vp, C.c_double, C.c_uint64, C.c_uint32]
        L.oracle_keep.restype = vp
        L.oracle_keep.argtypes = [vp, i, i]
        L.oracle_gelu_forward.argtypes = [vp, vp, sz]
        L.oracle_gelu_backward.argtypes = [vp, vp, vp, sz]
        L.oracle_crossentropy_forward.restype = r
        L.oracle_crossentropy_forward.argtypes = [vp, vp, vp, vp, i, i, i]
        L.oracle_crossentropy_backward.argtypes = [vp, vp, vp, i, i, i]
        L.oracle_adamw.argtypes = [vp, vp, vp, vp, sz, r, r, r, r, r, i]
        L.oracle_create.restype = vp
        L.oracle_create.argtypes = [i, i, i, i, i, i, i, i]
        L.oracle_free.argtypes = [vp]
        L.oracle_forward.restype = r
        L.oracle_forward.argtypes = [vp, vp, vp, vp]
        L.oracle_backward.restype = i
        L.oracle_backward.argtypes = [vp, vp, vp]
        L.oracle_adamw_model.argtypes = [vp, vp, vp, vp, vp, r, r, r, r, r, i]
        for name in ("oracle_logits", "oracle_probs", "oracle_losses"):
            getattr(L, name).restype = vp
            getattr(L, name).argtypes = [vp]
        L.oracle_act.restype = vp
        L.oracle_act.argtypes = [vp, i, i]

    # ---- helpers -------------------------------------------------------
    def arr(self, a):
        return np.ascontiguousarray(a, dtype=self.dtype)

    def num_threads(self):
        return self.lib.oracle_num_threads()

    def num_params(self, V, maxT, L, C_):
        return self.lib.oracle_num_params(V, maxT, L, C_)

    def param_sizes(self, V, maxT, L, C_):
        s = np.zeros(NTENSORS, dtype=np.uint64)
        self.lib.oracle_param_sizes(V, maxT, L, C_, _ptr(s))
        return [int(x) for x in s]

    # ---- layers (return new arrays; backward ones return fresh grads) --
    def encoder_forward(self, tok, wte, wpe):
        tok = np.ascontiguousarray(tok, dtype=np.int32)
        B, T = tok.shape
        Cc = wte.shape[1]
        x = np.zeros((B, T, Cc), dtype=self.dtype)
        self.lib.oracle_encoder_forward(_ptr(x), _ptr(tok), _ptr(self.arr(wte)),
                                        _ptr(self.arr(wpe)), B, T, Cc)
        return x

    def encoder_backward(self, dx, tok, V, maxT):
        tok = np.ascontiguousarray(tok, dtype=np.int32)
        B, T = tok.shape
        Cc = dx.shape[-1]
        dwte = np.zeros((V, Cc), dtype=self.dtype)
        dwpe = np.zeros((maxT, Cc), dtype=self.dtype)
        self.lib.oracle_encoder_backward(_ptr(dwte), _ptr(dwpe), _ptr(self.arr(dx)), _ptr(tok),
                                         B, T, Cc)
        return dwte, dwpe

    def layernorm_forward(self, x, w, b):
        x = self.arr(x)
        N, Cc = x.reshape(-1, x.shape[-1]).shape
        y = np.zeros_like(x)
        mean = np.zeros(N, dtype=self.dtype)
        rstd = np.zeros(N, dtype=self.dtype)
        self.lib.oracle_layernorm_forward(_ptr(y), _ptr(mean), _ptr(rstd), _ptr(x),
                                          _ptr(self.arr(w)), _ptr(self.arr(b)), N, Cc)
        return y, mean, rstd

    def layernorm_backward(self, dy, x, w, mean, rstd):
        x = self.arr(x)
        N, Cc = x.reshape(-1, x.shape[-1]).shape
        dx = np.zeros_like(x)
        dw = np.zeros(Cc, dtype=self.dtype)
        db = np.zeros(Cc, dtype=self.dtype)
        self.lib.oracle_layernorm_backward(_ptr(dx), _ptr(dw), _ptr(db), _ptr(self.arr(dy)),
                                           _ptr(x), _ptr(self.arr(w)), _ptr(self.arr(mean)),
                                           _ptr(self.arr(rstd)), N, Cc)
        return dx, dw, db

    def matmul_forward(self, x, w, bias=None):
        x = self.arr(x)
        OC, IC = w.shape
        N = x.size // IC
        y = np.zeros((N, OC), dtype=self.dtype)
        self.lib.oracle_matmul_forward(_ptr(y), _ptr(x), _ptr(self.arr(w)),
                                       _ptr(self.arr(bias)) if bias is not None else None,
                                       N, IC, OC)
        return y

    def matmul_backward(self, dy, x, w, with_bias=True):
        x = self.arr(x)
        OC, IC = w.shape
        N = x.size // IC
        dx = np.zeros((N, IC), dtype=self.dtype)
        dw = np.zeros((OC, IC), dtype=self.dtype)
        db = np.zeros(OC, dtype=self.dtype) if with_bias else None
        self.lib.oracle_matmul_backward(_ptr(dx), _ptr(dw), _ptr(db), _ptr(self.arr(dy)),
                                        _ptr(x), _ptr(self.arr(w)), N, IC, OC)
        return dx, dw, db

    def attention_forward(self, qkv, NH, keep=None, p=0.0):
        """keep: optional uint8 flags [B,NH,T,T] of attention dropout with probability p."""
        qkv = self.arr(qkv)
        B, T, C3 = qkv.shape
        Cc = C3 // 3
        y = np.zeros((B, T, Cc), dtype=self.dtype)
        P = np.zeros((B, NH, T, T), dtype=self.dtype)
        if keep is None:
            self.lib.oracle_attention_forward(_ptr(y), _ptr(P), _ptr(qkv), B, T, Cc, NH)
        else:
            keep = np.ascontiguousarray(keep, dtype=np.uint8)
            assert keep.size == B * NH * T * T
            self.lib.oracle_attention_forward_dropout(_ptr(y), _ptr(P), _ptr(qkv), B, T, Cc, NH,
                                                      _ptr(keep), float(p))
        return y, P

    def attention_backward(self, dy, qkv, P, NH, keep=None, p=0.0):
        qkv = self.arr(qkv)
        B, T, C3 = qkv.shape
        dqkv = np.zeros_like(qkv)
        if keep is None:
            self.lib.oracle_attention_backward(_ptr(dqkv), _ptr(self.arr(dy)), _ptr(qkv),
                                               _ptr(self.arr(P)), B, T, C3 // 3, NH)
        else:
            keep = np.ascontiguousarray(keep, dtype=np.uint8)
            self.lib.oracle_attention_backward_dropout(_ptr(dqkv), _ptr(self.arr(dy)), _ptr(qkv),
                                                       _ptr(self.arr(P)), B, T, C3 // 3, NH,
                                                       _ptr(keep), float(p))
        return dqkv

    # ---- dropout ------------------------------------------------------
    def philox(self, ctr, key):
        """Philox4x32-10 of one counter (4 words) under one key (2 words)."""
        c = np.ascontiguousarray(ctr, dtype=np.uint32)
        k = np.ascontiguousarray(key, dtype=np.uint32)
        assert c.size == 4 and k.size == 2
        out = np.zeros(4, dtype=np.uint32)
        self.lib.oracle_philox4x32_10(_ptr(out), _ptr(c), _ptr(k))
        return out

    def dropout_keep(self, n, seed, site, step, p):
        """uint8 keep flags of elements 0..n-1 of one dropout site."""
        keep = np.zeros(int(n), dtype=np.uint8)
        self.lib.oracle_dropout_keep(_ptr(keep), int(n), int(seed), int(site), int(step), float(p))
        return keep

    def dropout_apply(self, x, keep, p):
        x = self.arr(x)
        keep = np.ascontiguousarray(keep, dtype=np.uint8)
        assert keep.size == x.size
        y = np.zeros_like(x)
        self.lib.oracle_dropout_apply(_ptr(y), _ptr(x), _ptr(keep), x.size, float(p))
        return y

    def gelu_forward(self, x):
        x = self.arr(x)
        y = np.zeros_like(x)
        self.lib.oracle_gelu_forward(_ptr(y), _ptr(x), x.size)
        return y

    def gelu_backward(self, x, dy):
        x = self.arr(x)
        dx = np.zeros_like(x)
        self.lib.oracle_gelu_backward(_ptr(dx), _ptr(x), _ptr(self.arr(dy)), x.size)
        return dx

    def crossentropy_forward(self, z, tgt, V=None):
        z = self.arr(z)
        N, ld = z.shape
        V = V or ld
        tgt = np.ascontiguousarray(tgt, dtype=np.int32).reshape(-1)
        losses = np.zeros(N, dtype=self.dtype)
        probs = np.zeros((N, V), dtype=self.dtype)
        mean = self.lib.oracle_crossentropy_forward(_ptr(losses), _ptr(probs), _ptr(z),
                                                    _ptr(tgt), N, V, ld)
        return mean, losses, probs

    def crossentropy_backward(self, probs, tgt, ld=None):
        probs = self.arr(probs)
        N, V = probs.shape
        ld = ld or V
        tgt = np.ascontiguousarray(tgt, dtype=np.int32).reshape(-1)
        dz = np.zeros((N, ld), dtype=self.dtype)
        self.lib.oracle_crossentropy_backward(_ptr(dz), _ptr(probs), _ptr(tgt), N, V, ld)
        return dz

    def adamw(self, p, g, m, v, lr, b1, b2, eps, wd, t):
        """In-place on p, m, v (arrays of the build's dtype)."""
        for a in (p, g, m, v):
            assert a.dtype == self.dtype and a.flags.c_contiguous
        self.lib.oracle_adamw(_ptr(p), _ptr(g), _ptr(m), _ptr(v), p.size, lr, b1, b2, eps, wd, t)

    def model(self, cfg, B, T, last_only=False):
        return OracleModel(self, cfg, B, T, last_only)


class OracleModel:
    """One oracle model instance for a fixed (B, T).

    ``cfg`` is a mapping with V, maxT, L, H (heads) and C.
    """

    def __init__(self, oracle, cfg, B, T, last_only=False):
        self.o = oracle
        self.cfg = dict(cfg)
        self.B, self.T = B, T
        self.last_only = bool(last_only)
        c = self.cfg
        self.h = oracle.lib.oracle_create(c["V"], c["maxT"], c["L"], c["H"], c["C"], B, T,
                                          int(last_only))
        if not self.h:
            raise ValueError("oracle_create rejected the configuration")
        self.nparams = oracle.num_params(c["V"], c["maxT"], c["L"], c["C"])

    def __del__(self):
        h = getattr(self, "h", None)
        if h:
            self.o.lib.oracle_free(h)
            self.h = None

    def forward(self, params, tok, tgt=None):
        assert params.dtype == self.o.dtype and params.size == self.nparams
        tok = np.ascontiguousarray(tok, dtype=np.int32)
        assert tok.shape == (self.B, self.T)
        tgt_arr = None
        if tgt is not None:
            tgt_arr = np.ascontiguousarray(tgt, dtype=np.int32)
            assert tgt_arr.shape == (self.B, self.T)
        return float(self.o.lib.oracle_forward(self.h, _ptr(params), _ptr(tok), _ptr(tgt_arr)))

    def set_dropout(self, p, seed=0, step=0):
        """Dropout for the following forwards (p < 0 turns it off)."""
        if self.o.lib.oracle_set_dropout(self.h, float(p), int(seed), int(step)) != 0:
            raise ValueError("oracle_set_dropout: p must be below 1")

    def keep(self, which, layer=0):
        """Keep flags of the last forward: 'emb', 'att' [B,NH,T,T], 'attproj', 'fcproj'."""
        c = self.cfg
        N = self.B * self.T
        idx = {"emb": 0, "att": 1, "attproj": 2, "fcproj": 3}[which]
        n = self.B * c["H"] * self.T * self.T if which == "att" else N * c["C"]
        addr = self.o.lib.oracle_keep(self.h, idx, layer)
        if not addr:
            return None
        return np.frombuffer((C.c_uint8 * n).from_address(addr), dtype=np.uint8, count=n).copy()

    def backward(self, params):
        grads = np.zeros(self.nparams, dtype=self.o.dtype)
        rc = self.o.lib.oracle_backward(self.h, _ptr(params), _ptr(grads))
        if rc != 0:
            raise RuntimeError("oracle_backward needs a full forward with targets first")
        return grads

    def adamw(self, params, grads, m, v, lr, b1, b2, eps, wd, t):
        for a in (params, grads, m, v):
            assert a.dtype == self.o.dtype and a.size == self.nparams
        self.o.lib.oracle_adamw_model(self.h, _ptr(params), _ptr(grads), _ptr(m), _ptr(v),
                                      lr, b1, b2, eps, wd, t)

    def _view(self, addr, n):
        buf = (self.o.ctreal * n).from_address(addr)
        return np.frombuffer(buf, dtype=self.o.dtype, count=n).copy()

    def rows(self):
        return self.B if self.last_only else self.B * self.T

    def logits(self):
        V = self.cfg["V"]
        return self._view(self.o.lib.oracle_logits(self.h), self.rows() * V).reshape(-1, V)

    def probs(self):
        V = self.cfg["V"]
        return self._view(self.o.lib.oracle_probs(self.h), self.rows() * V).reshape(-1, V)

    def losses(self):
        return self._view(self.o.lib.oracle_losses(self.h), self.rows())

    def act(self, name, layer=0):
        c = self.cfg
        N = self.B * self.T
        shapes = {"x0": (N, c["C"]), "ln1": (N, c["C"]), "qkv": (N, 3 * c["C"]),
                  "atty": (N, c["C"]), "res2": (N, c["C"]), "ln2": (N, c["C"]),
                  "h": (N, 4 * c["C"]), "g": (N, 4 * c["C"]), "res3": (N, c["C"]),
                  "lnf": (N, c["C"]), "P": (self.B, c["H"], self.T, self.T),
                  "ln1_mean": (N,), "ln1_rstd": (N,)}
        shp = shapes[name]
        n = int(np.prod(shp))
        return self._view(self.o.lib.oracle_act(self.h, ACT[name], layer), n).reshape(shp)


def sample_topk(logits, k, u):
    """Top-k sampling of each row ("GPT-2 from scratch with torch", section
    生成样本): keep the k highest scores, turn them into probabilities with a
    softmax, and draw from them; the draw is the caller's uniform number u[n] in
    [0, 1), applied as an inverse cumulative distribution over the kept tokens in
    ascending index order (the order in which a multinomial draw over the whole
    vocabulary walks the tokens).  Ties at the cut keep the lower index; NaN
    scores are never kept.  Plain loops in float64.  Returns (tokens, cumulative
    boundaries per row) so that tests can tell draws that sit on a boundary."""
    import math
    z = np.asarray(logits, dtype=np.float64)
    N, V = z.shape
    out = np.zeros(N, dtype=np.int32)
    bounds = []
    for n in range(N):
        cand = [v for v in range(V) if z[n, v] == z[n, v]]
        cand.sort(key=lambda v: (-z[n, v], v))
        keep = sorted(cand[:k])
        if not keep:
            bounds.append([])
            continue
        zmax = max(z[n, v] for v in keep)
        p = [math.exp(z[n, v] - zmax) for v in keep]
        s = sum(p)
        cum, c = [], 0.0
        out[n] = keep[-1]
        chosen = False
        for v, pv in zip(keep, p):
            c += pv / s
            cum.append(c)
            if not chosen and c > u[n]:
                out[n] = v
                chosen = True
        bounds.append(cum)
    return out, bounds


def split_params(flat, sizes):
    """Views of the 16 tensors of a flat parameter array, by name."""
    out, off = {}, 0
    for name, s in zip(TENSOR_NAMES, sizes):
        out[name] = flat[off:off + s]
        off += s
    return out
