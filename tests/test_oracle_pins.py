"""Pins for the CPU oracle: values the pages print, closed forms, invariants,
library routines and brute force -- never the oracle's own formula retyped.

Each test targets a mistake the oracle could plausibly contain (a dropped
term, a wrong sign or index, a transposed operand, a missing mask).
"""
import math

import numpy as np
import pytest

from conftest import read_golden
from gpt_decoder_step_train_b300 import synthetic as syn
from oracle import split_params

TINY = syn.CONFIGS["tiny"]


def tiny_inputs(cfg=TINY, seed=None):
    params = syn.init_params(cfg, seed=seed).astype(np.float64)
    tok, tgt = syn.draw_tokens(cfg)
    return params, tok, tgt


# ---------------------------------------------------------------- printed values

def test_param_count_matches_run_log(o64):
    g = read_golden("gpt2_124m_run_log.txt")
    cfg = syn.CONFIGS["124M"]
    assert (cfg.V, cfg.maxT, cfg.L, cfg.H, cfg.C) == (
        g["vocab_size"], g["max_seq_len"], g["num_layers"], g["num_heads"], g["channels"])
    n = o64.num_params(cfg.V, cfg.maxT, cfg.L, cfg.C)
    assert n == g["num_parameters"] == syn.num_params(cfg)
    # an untied lm_head would add V*C parameters and miss the printed count
    assert n + cfg.V * cfg.C != g["num_parameters"]


def test_activation_count_of_run_log_fixes_the_small_batch_shape():
    """The run log prints num_activations = 73,323,776: the floats of the C
    trainer's per-layer activation tensors (LayerNorm outputs and statistics,
    qkv, attention scores and probabilities, one T x T matrix each per head,
    attention output and projection, residuals, the MLP's pre-activation and
    GELU output, its projection), the final LayerNorm, logits, probabilities and
    losses.  With the model's widths (qkv 3C, MLP 4C, V unpadded) the count
    holds for B = 4 sequences of T = 64 positions, the small 124M configuration,
    and for no other batch shape of up to 4096 positions."""
    g = read_golden("gpt2_124m_run_log.txt")
    cfg = syn.CONFIGS["124M_small"]
    L, C, H, V = cfg.L, cfg.C, cfg.H, cfg.V

    def count(B, T):
        N = B * T
        per_layer = (N * C + 2 * N            # ln_1 output, mean, rstd
                     + N * 3 * C              # qkv
                     + 2 * B * H * T * T      # scores, probabilities
                     + N * C + N * C          # attention output, its projection
                     + N * C                  # residual after attention
                     + N * C + 2 * N          # ln_2 output, mean, rstd
                     + 2 * N * 4 * C          # MLP pre-activation, GELU output
                     + N * C + N * C)         # MLP projection, block output
        return N * C + L * per_layer + N * C + 2 * N + 2 * N * V + N

    assert count(cfg.B, cfg.T) == g["num_activations"]
    others = [(B, T) for B in range(1, 65) for T in range(1, 1025)
              if B * T <= 4096 and (B, T) != (cfg.B, cfg.T) and count(B, T) == g["num_activations"]]
    assert others == []


def test_uniform_logits_give_printed_loss(o64):
    """wte = 0 makes every tied logit exactly 0, so the loss is exactly ln V."""
    g = read_golden("uniform_char_loss.txt")
    assert TINY.V == g["vocab_size"]
    params, tok, tgt = tiny_inputs()
    sizes = o64.param_sizes(TINY.V, TINY.maxT, TINY.L, TINY.C)
    split_params(params, sizes)["wte"][:] = 0.0
    m = o64.model(TINY.dims(), TINY.B, TINY.T)
    loss = m.forward(params, tok, tgt)
    assert np.all(m.logits() == 0.0)
    assert abs(loss - math.log(TINY.V)) < 1e-12
    assert round(loss, int(g["decimals"])) == g["loss"]


def test_uniform_logits_dlogits_closed_form(o64):
    N, V = 10, 65
    z = np.zeros((N, V))
    tgt = np.arange(N) * 7 % V
    mean, losses, probs = o64.crossentropy_forward(z, tgt)
    dz = o64.crossentropy_backward(probs, tgt)
    want = np.full((N, V), 1.0 / V / N)
    want[np.arange(N), tgt] -= 1.0 / N
    assert np.abs(dz - want).max() < 1e-15
    assert abs(mean - math.log(V)) < 1e-12


def test_init_loss_close_to_ln_V(o64):
    params, tok, tgt = tiny_inputs()
    loss = o64.model(TINY.dims(), TINY.B, TINY.T).forward(params, tok, tgt)
    # N(0, 0.02) init keeps logits tiny: loss = ln V + O(var(z))
    assert math.log(TINY.V) < loss < math.log(TINY.V) + 0.05


def test_gelu_constants_match_page(o64):
    g = read_golden("gelu_tanh_constants.txt")
    s = math.sqrt(2 / math.pi)
    assert abs(s - g["sqrt_2_over_pi_truncated"]) < 1e-7
    # gelu(x) - x = -0.5 x (1 - tanh(u)); at x=1 this isolates the cubic coefficient
    x = np.array([1.0])
    y = o64.gelu_forward(x)[0]
    u = math.atanh(2 * y - 1)
    assert abs(u / s - (1 + g["cubic_coefficient"])) < 1e-12


def test_layernorm_eps_matches_page(o64):
    g = read_golden("layernorm_eps.txt")
    # a constant row has variance 0, so rstd = 1/sqrt(eps)
    x = np.full((1, 8), 3.0)
    _, mean, rstd = o64.layernorm_forward(x, np.ones(8), np.zeros(8))
    assert mean[0] == 3.0
    assert abs(rstd[0] - 1 / math.sqrt(g["eps"])) < 1e-9


# ---------------------------------------------------------------- invariants

def test_softmax_rows_sum_to_one(o64):
    rng = np.random.default_rng(3)
    z = rng.normal(size=(17, 101)) * 5
    tgt = rng.integers(0, 101, 17)
    mean, losses, probs = o64.crossentropy_forward(z, tgt)
    assert np.abs(probs.sum(1) - 1).max() < 1e-14
    # lse - z[tgt] against scipy's logsumexp
    from scipy.special import logsumexp
    assert np.abs(losses - (logsumexp(z, axis=1) - z[np.arange(17), tgt])).max() < 1e-12


def test_crossentropy_padded_stride_ignores_tail(o64):
    rng = np.random.default_rng(4)
    z = rng.normal(size=(5, 13))
    zp = np.concatenate([z, np.full((5, 3), 1e30)], axis=1)   # garbage past V
    tgt = rng.integers(0, 13, 5)
    a = o64.crossentropy_forward(z, tgt)[1]
    b = o64.crossentropy_forward(zp, tgt, V=13)[1]
    assert np.array_equal(a, b)


def test_layernorm_normalises_before_affine(o64):
    rng = np.random.default_rng(5)
    x = rng.normal(size=(9, 77)) * 3 + 1.5
    y, mean, rstd = o64.layernorm_forward(x, np.ones(77), np.zeros(77))
    assert np.abs(y.mean(1)).max() < 1e-14
    var = x.var(1)
    assert np.abs(y.var(1) - var / (var + 1e-5)).max() < 1e-12
    assert np.abs(mean - x.mean(1)).max() < 1e-14
    # affine applies per column
    w, b = rng.normal(size=77), rng.normal(size=77)
    y2 = o64.layernorm_forward(x, w, b)[0]
    assert np.abs(y2 - (y * w + b)).max() < 1e-12


def test_layernorm_backward_sums_to_zero_and_matches_fd(o64):
    rng = np.random.default_rng(6)
    N, Cc = 4, 11
    x = rng.normal(size=(N, Cc))
    w, b = rng.normal(size=Cc), rng.normal(size=Cc)
    dy = rng.normal(size=(N, Cc))
    _, mean, rstd = o64.layernorm_forward(x, w, b)
    dx, dw, db = o64.layernorm_backward(dy, x, w, mean, rstd)
    _, _, _ = o64.layernorm_backward(dy, x, np.ones(Cc), mean, rstd)
    dx1 = o64.layernorm_backward(dy, x, np.ones(Cc), mean, rstd)[0]
    assert np.abs(dx1.sum(1)).max() < 1e-12      # shift invariance of LN
    # brute-force central differences of sum(dy * y)
    f = lambda xx, ww, bb: float((o64.layernorm_forward(xx, ww, bb)[0] * dy).sum())
    h = 1e-6
    for arr, grad in ((x, dx), (w, dw), (b, db)):
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            a0 = arr[i]
            arr[i] = a0 + h; fp = f(x, w, b)
            arr[i] = a0 - h; fm = f(x, w, b)
            arr[i] = a0
            fd[i] = (fp - fm) / (2 * h)
        assert np.abs(fd - grad).max() < 1e-7 * max(1.0, np.abs(grad).max())


def test_attention_zero_queries_is_running_mean(o64):
    """Q = 0 gives equal weights over the causal window: O_i = mean_{j<=i} V_j
    (the lower-triangular averaging identity)."""
    rng = np.random.default_rng(7)
    B, T, Cc, NH = 2, 9, 12, 3
    qkv = rng.normal(size=(B, T, 3 * Cc))
    qkv[:, :, :Cc] = 0.0
    y, P = o64.attention_forward(qkv, NH)
    v = qkv[:, :, 2 * Cc:]
    want = np.cumsum(v, axis=1) / np.arange(1, T + 1)[None, :, None]
    assert np.abs(y - want).max() < 1e-14
    tril = np.tril(np.ones((T, T))) / np.arange(1, T + 1)[:, None]
    assert np.abs(P - tril).max() < 1e-15


def test_attention_single_position_returns_values(o64):
    rng = np.random.default_rng(8)
    qkv = rng.normal(size=(3, 1, 3 * 8))
    y, _ = o64.attention_forward(qkv, 2)
    assert np.array_equal(y, qkv[:, :, 16:])


def test_attention_matches_dense_library_formula(o64):
    """Per head: softmax(mask(QK^T/sqrt(hs))) V with numpy matmuls and a
    triangular mask, heads laid side by side."""
    rng = np.random.default_rng(9)
    B, T, Cc, NH = 2, 13, 24, 4
    hs = Cc // NH
    qkv = rng.normal(size=(B, T, 3 * Cc))
    y, P = o64.attention_forward(qkv, NH)
    q, k, v = (qkv[:, :, i * Cc:(i + 1) * Cc].reshape(B, T, NH, hs).transpose(0, 2, 1, 3)
               for i in range(3))
    s = q @ k.transpose(0, 1, 3, 2) / math.sqrt(hs)
    s = np.where(np.tril(np.ones((T, T), dtype=bool)), s, -np.inf)
    from scipy.special import softmax
    p = softmax(s, axis=-1)
    want = (p @ v).transpose(0, 2, 1, 3).reshape(B, T, Cc)
    assert np.abs(y - want).max() < 1e-13
    assert np.abs(P - p).max() < 1e-14


def test_causal_invariance_of_full_model(o64):
    params, tok, tgt = tiny_inputs()
    m = o64.model(TINY.dims(), TINY.B, TINY.T)
    m.forward(params, tok, tgt)
    z0 = m.logits().reshape(TINY.B, TINY.T, -1)
    t = 11
    tok2 = tok.copy()
    tok2[:, t + 1:] = (tok2[:, t + 1:] + 5) % TINY.V
    m.forward(params, tok2, tgt)
    z1 = m.logits().reshape(TINY.B, TINY.T, -1)
    assert np.array_equal(z0[:, :t + 1], z1[:, :t + 1])
    assert not np.array_equal(z0[:, t + 1:], z1[:, t + 1:])


def test_last_only_forward_matches_full_rows(o64):
    params, tok, tgt = tiny_inputs()
    full = o64.model(TINY.dims(), TINY.B, TINY.T)
    full.forward(params, tok, tgt)
    last = o64.model(TINY.dims(), TINY.B, TINY.T, last_only=True)
    last.forward(params, tok, tgt)
    zf = full.logits().reshape(TINY.B, TINY.T, -1)[:, -1]
    assert np.array_equal(zf, last.logits())
    assert np.array_equal(full.losses().reshape(TINY.B, TINY.T)[:, -1], last.losses())


# ---------------------------------------------------------------- GELU

def test_gelu_special_values(o64):
    x = np.array([0.0, 12.0, -12.0, 1e-8])
    y = o64.gelu_forward(x)
    assert y[0] == 0.0
    assert abs(y[1] - 12.0) < 1e-12 and abs(y[2]) < 1e-12
    d = o64.gelu_backward(np.array([0.0]), np.array([1.0]))
    assert d[0] == 0.5


def test_gelu_close_to_exact_erf_form(o64):
    x = np.linspace(-6, 6, 2001)
    y = o64.gelu_forward(x)
    exact = np.array([v * 0.5 * (1 + math.erf(v / math.sqrt(2))) for v in x])
    assert np.abs(y - exact).max() < 1e-3


def test_gelu_backward_matches_fd(o64):
    x = np.linspace(-5, 5, 101)
    d = o64.gelu_backward(x, np.ones_like(x))
    h = 1e-6
    fd = (o64.gelu_forward(x + h) - o64.gelu_forward(x - h)) / (2 * h)
    assert np.abs(d - fd).max() < 1e-8


# ---------------------------------------------------------------- linear algebra

def test_matmul_matches_numpy(o64):
    rng = np.random.default_rng(10)
    N, IC, OC = 7, 13, 5
    x, w, b = rng.normal(size=(N, IC)), rng.normal(size=(OC, IC)), rng.normal(size=OC)
    y = o64.matmul_forward(x, w, b)
    assert np.abs(y - (x @ w.T + b)).max() < 1e-12
    assert np.abs(o64.matmul_forward(x, w) - x @ w.T).max() < 1e-12
    dy = rng.normal(size=(N, OC))
    dx, dw, db = o64.matmul_backward(dy, x, w)
    assert np.abs(dx - dy @ w).max() < 1e-12
    assert np.abs(dw - dy.T @ x).max() < 1e-12
    assert np.abs(db - dy.sum(0)).max() < 1e-12


def test_encoder_forward_bit_exact_gather(o32):
    rng = np.random.default_rng(11)
    V, maxT, Cc, B, T = 50, 16, 8, 3, 10
    wte = rng.normal(size=(V, Cc)).astype(np.float32)
    wpe = rng.normal(size=(maxT, Cc)).astype(np.float32)
    tok = rng.integers(0, V, (B, T)).astype(np.int32)
    x = o32.encoder_forward(tok, wte, wpe)
    assert np.array_equal(x, wte[tok] + wpe[None, :T])


def test_encoder_backward_is_scatter_add(o64):
    rng = np.random.default_rng(12)
    V, maxT, Cc, B, T = 9, 12, 4, 3, 7
    tok = rng.integers(0, V, (B, T)).astype(np.int32)
    dx = rng.normal(size=(B, T, Cc))
    dwte, dwpe = o64.encoder_backward(dx, tok, V, maxT)
    want = np.zeros((V, Cc))
    np.add.at(want, tok.reshape(-1), dx.reshape(-1, Cc))
    assert np.abs(dwte - want).max() < 1e-13
    assert np.abs(dwpe[:T] - dx.sum(0)).max() < 1e-13
    assert np.all(dwpe[T:] == 0)


# ---------------------------------------------------------------- AdamW

def test_adamw_first_step_closed_form(o64):
    rng = np.random.default_rng(13)
    n = 1000
    p0 = rng.normal(size=n)
    g = rng.normal(size=n) * 1e-3
    g[:10] = 0.0
    lr, wd, eps = 1e-3, 0.1, 1e-8
    for decay in (0.0, wd):
        p, m, v = p0.copy(), np.zeros(n), np.zeros(n)
        o64.adamw(p, g, m, v, lr, 0.9, 0.999, eps, decay, 1)
        # t = 1: mhat = g, vhat = g^2
        want = p0 - lr * (g / (np.abs(g) + eps) + decay * p0)
        assert np.abs(p - want).max() < 1e-15
        if decay == 0.0:
            assert np.array_equal(p[:10], p0[:10])


def test_adamw_model_decays_only_2d_tensors(o64):
    params, tok, tgt = tiny_inputs()
    sizes = o64.param_sizes(TINY.V, TINY.maxT, TINY.L, TINY.C)
    m = o64.model(TINY.dims(), TINY.B, TINY.T)
    zero = np.zeros_like(params)
    p = params.copy()
    m.adamw(p, zero, zero.copy(), zero.copy(), 1e-2, 0.9, 0.999, 1e-8, 0.5, 1)
    before, after = split_params(params, sizes), split_params(p, sizes)
    for name in before:
        if name in ("wte", "wpe", "qkvw", "attprojw", "fcw", "fcprojw"):
            assert np.allclose(after[name], before[name] * (1 - 1e-2 * 0.5), rtol=0, atol=1e-15)
        else:
            assert np.array_equal(after[name], before[name])


# ---------------------------------------------------------------- whole backward

def _loss(o, cfg, params, tok, tgt):
    return o.model(cfg.dims(), tok.shape[0], tok.shape[1]).forward(params, tok, tgt)


def test_gradcheck_finite_differences_tiny(o64):
    """FP64 central differences on sampled parameters of every tensor."""
    params, tok, tgt = tiny_inputs()
    m = o64.model(TINY.dims(), TINY.B, TINY.T)
    m.forward(params, tok, tgt)
    grads = m.backward(params)
    sizes = o64.param_sizes(TINY.V, TINY.maxT, TINY.L, TINY.C)
    rng = np.random.default_rng(14)
    offs = np.concatenate([[0], np.cumsum(sizes)])
    idx = []
    for i in range(16):
        idx += list(rng.integers(offs[i], offs[i + 1], 12))
    # rows of wte that never occur as input tokens still get the lm_head gradient;
    # rows of wpe at positions >= T must have exactly zero gradient
    idx += [int(offs[1] + TINY.T * TINY.C + 3), int(offs[1] + (TINY.maxT - 1) * TINY.C)]
    h = 1e-5
    worst = 0.0
    for i in idx:
        p0 = params[i]
        params[i] = p0 + h; lp = m.forward(params, tok, tgt)
        params[i] = p0 - h; lm = m.forward(params, tok, tgt)
        params[i] = p0
        fd = (lp - lm) / (2 * h)
        err = abs(fd - grads[i])
        worst = max(worst, err / (abs(grads[i]) + 1e-6))
        assert err <= 1e-6 * abs(grads[i]) + 1e-9, (i, fd, grads[i])
    assert grads[idx[-1]] == 0.0 and grads[idx[-2]] == 0.0


def test_gradcheck_directional_all_params(o64):
    params, tok, tgt = tiny_inputs()
    m = o64.model(TINY.dims(), TINY.B, TINY.T)
    m.forward(params, tok, tgt)
    grads = m.backward(params)
    rng = np.random.default_rng(15)
    for _ in range(3):
        d = rng.normal(size=params.size)
        h = 1e-6
        f = lambda s: m.forward(params + s * h * d, tok, tgt)
        # fourth-order central difference: truncation error O(h^4)
        fd = (-f(2) + 8 * f(1) - 8 * f(-1) + f(-2)) / (12 * h)
        assert abs(fd - grads @ d) <= 1e-6 * abs(grads @ d) + 1e-9


def _torch_model_step(cfg, params, tok, tgt, steps, lr, wd):
    """Second opinion: the same architecture written with torch.nn.functional in
    float64, differentiated by autograd and updated by torch.optim.AdamW."""
    import torch
    import torch.nn.functional as F
    shapes = syn.tensor_shapes(cfg)
    ts, off = {}, 0
    for name in syn.TENSOR_NAMES:
        n = int(np.prod(shapes[name]))
        ts[name] = torch.tensor(params[off:off + n].reshape(shapes[name]), dtype=torch.float64,
                                requires_grad=True)
        off += n
    decay_names = ("wte", "wpe", "qkvw", "attprojw", "fcw", "fcprojw")
    decay = [ts[k] for k in decay_names]
    rest = [ts[k] for k in syn.TENSOR_NAMES if k not in decay_names]
    opt = torch.optim.AdamW([{"params": decay, "weight_decay": wd},
                             {"params": rest, "weight_decay": 0.0}],
                            lr=lr, betas=(0.9, 0.999), eps=1e-8)
    tok_t = torch.tensor(tok, dtype=torch.long)
    tgt_t = torch.tensor(tgt, dtype=torch.long)
    B, T = tok.shape
    Cc, H, V = cfg.C, cfg.H, cfg.V
    hs = Cc // H
    losses, grads = [], None
    for _ in range(steps):
        opt.zero_grad()
        x = ts["wte"][tok_t] + ts["wpe"][:T]
        for l in range(cfg.L):
            a = F.layer_norm(x, (Cc,), ts["ln1w"][l], ts["ln1b"][l], eps=1e-5)
            qkv = F.linear(a, ts["qkvw"][l], ts["qkvb"][l])
            q, k, v = (z.view(B, T, H, hs).transpose(1, 2) for z in qkv.split(Cc, dim=-1))
            att = F.scaled_dot_product_attention(q, k, v, is_causal=True)
            att = att.transpose(1, 2).reshape(B, T, Cc)
            x = x + F.linear(att, ts["attprojw"][l], ts["attprojb"][l])
            a = F.layer_norm(x, (Cc,), ts["ln2w"][l], ts["ln2b"][l], eps=1e-5)
            hmid = F.gelu(F.linear(a, ts["fcw"][l], ts["fcb"][l]), approximate="tanh")
            x = x + F.linear(hmid, ts["fcprojw"][l], ts["fcprojb"][l])
        x = F.layer_norm(x, (Cc,), ts["lnfw"], ts["lnfb"], eps=1e-5)
        logits = x @ ts["wte"].T
        loss = F.cross_entropy(logits.reshape(-1, V), tgt_t.reshape(-1))
        loss.backward()
        if grads is None:
            grads = np.concatenate([ts[k].grad.detach().numpy().reshape(-1)
                                    for k in syn.TENSOR_NAMES])
        losses.append(float(loss.detach()))
        opt.step()
    newp = np.concatenate([ts[k].detach().numpy().reshape(-1) for k in syn.TENSOR_NAMES])
    return losses, grads, newp


@pytest.mark.parametrize("cfg", [
    TINY,
    # ragged: head size 8, T not a power of two, odd vocabulary, 3 layers
    syn.Config("ragged", V=97, maxT=24, L=3, H=6, C=48, B=3, T=19, lr=3e-3, wd=0.1),
])
def test_full_step_matches_torch_autograd(o64, cfg):
    params = syn.init_params(cfg).astype(np.float64)
    tok, tgt = syn.draw_tokens(cfg)
    steps = 3
    t_losses, t_grads, t_params = _torch_model_step(cfg, params, tok, tgt, steps, cfg.lr, cfg.wd)
    m = o64.model(cfg.dims(), cfg.B, cfg.T)
    p = params.copy()
    am, av = np.zeros_like(p), np.zeros_like(p)
    for t in range(1, steps + 1):
        loss = m.forward(p, tok, tgt)
        assert abs(loss - t_losses[t - 1]) < 1e-12
        g = m.backward(p)
        if t == 1:
            assert np.abs(g - t_grads).max() < 1e-12 * max(1.0, np.abs(t_grads).max()) + 1e-15
        m.adamw(p, g, am, av, cfg.lr, 0.9, 0.999, 1e-8, cfg.wd, t)
    assert np.abs(p - t_params).max() < 1e-12


def test_overfit_one_batch_loss_falls_monotonically(o64):
    """Ten AdamW steps on one fixed batch (the train script's sanity run)."""
    params, tok, tgt = tiny_inputs()
    m = o64.model(TINY.dims(), TINY.B, TINY.T)
    am, av = np.zeros_like(params), np.zeros_like(params)
    losses = []
    for t in range(1, 11):
        losses.append(m.forward(params, tok, tgt))
        g = m.backward(params)
        m.adamw(params, g, am, av, TINY.lr, TINY.b1, TINY.b2, TINY.eps, TINY.wd, t)
    assert all(b < a for a, b in zip(losses, losses[1:])), losses


def test_float_build_tracks_double_build(o32, o64):
    params, tok, tgt = tiny_inputs()
    m64 = o64.model(TINY.dims(), TINY.B, TINY.T)
    m32 = o32.model(TINY.dims(), TINY.B, TINY.T)
    l64 = m64.forward(params, tok, tgt)
    l32 = m32.forward(params.astype(np.float32), tok, tgt)
    assert abs(l64 - l32) < 1e-5
    g64 = m64.backward(params)
    g32 = m32.backward(params.astype(np.float32))
    assert np.linalg.norm(g32 - g64) / np.linalg.norm(g64) < 1e-5


# ---- top-k sampling (generation: keep the k highest scores, softmax, draw) ----
def test_sample_topk_k1_is_argmax():
    from oracle import sample_topk
    rng = np.random.default_rng(11)
    z = rng.normal(size=(20, 300))
    tok, _ = sample_topk(z, 1, rng.random(20))
    assert np.array_equal(tok, np.argmax(z, axis=1))


def test_sample_topk_equal_scores_are_uniform_over_kept_indices():
    """k equal maxima: each kept token has probability 1/k, so u in [j/k, (j+1)/k)
    selects the j-th smallest kept index (closed form)."""
    from oracle import sample_topk
    V, k = 97, 4
    z = np.full((1, V), -3.0)
    kept = [5, 17, 60, 90]
    z[0, kept] = 2.5
    for j in range(k):
        for frac in (0.05, 0.5, 0.95):
            tok, _ = sample_topk(z, k, np.array([(j + frac) / k]))
            assert tok[0] == kept[j]


def test_sample_topk_two_tokens_closed_form_boundary():
    from oracle import sample_topk
    z = np.full((1, 10), -50.0)
    z[0, 7], z[0, 2] = 1.0, 0.25                      # kept in index order: 2 then 7
    p2 = np.exp(0.25) / (np.exp(0.25) + np.exp(1.0))
    assert sample_topk(z, 2, np.array([p2 - 1e-9]))[0][0] == 2
    assert sample_topk(z, 2, np.array([p2 + 1e-9]))[0][0] == 7
    assert sample_topk(z, 2, np.array([0.999999999]))[0][0] == 7


def test_sample_topk_tie_at_cut_keeps_lower_index_and_skips_nan():
    from oracle import sample_topk
    z = np.array([[3.0, 5.0, 3.0, 3.0, np.nan, 3.0]])
    # k = 2 keeps 1 (5.0) and 0 (the lowest-index 3.0); u near 1 picks the larger index kept
    tok, bounds = sample_topk(z, 2, np.array([0.999999]))
    assert tok[0] == 1 and len(bounds[0]) == 2
    tok, _ = sample_topk(z, 2, np.array([0.0]))
    assert tok[0] == 0
    tok, _ = sample_topk(np.array([[np.nan, np.nan, 1.0]]), 3, np.array([0.5]))
    assert tok[0] == 2


def test_sample_topk_frequencies_follow_the_kept_softmax():
    """Draws on a fine grid of u reproduce the softmax of the kept scores."""
    from oracle import sample_topk
    rng = np.random.default_rng(12)
    z = rng.normal(size=(1, 40)) * 2
    k = 6
    grid = (np.arange(4000) + 0.5) / 4000
    toks = np.array([sample_topk(z, k, np.array([g]))[0][0] for g in grid])
    kept = np.argsort(-z[0], kind="stable")[:k]
    p = np.exp(z[0, kept] - z[0, kept].max())
    p /= p.sum()
    for v, pv in zip(kept, p):
        assert abs(np.mean(toks == v) - pv) < 1e-3


# ---- dropout (inverted dropout at the four sites; Philox4x32-10 draws) ----
def _philox_kat():
    from conftest import GOLDEN
    import os
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if line:
                rows.append([int(w, 16) for w in line])
    return rows


def test_philox_known_answer_vectors(o64):
    rows = _philox_kat()
    assert len(rows) == 3
    for r in rows:
        assert list(o64.philox(r[0:4], r[4:6])) == r[6:10]


def test_dropout_keep_is_the_counter_word_against_the_threshold(o64):
    """Element e uses word e mod 4 of the draw at counter (e/4, 0, site, step);
    a word equal to the threshold is kept, one below it is dropped."""
    seed, site, step = 0x1234_5678_9ABC_DEF0, 7, 3
    key = [seed & 0xFFFFFFFF, seed >> 32]
    n = 37
    words = np.concatenate([o64.philox([q, 0, site, step], key) for q in range((n + 3) // 4)])[:n]
    w = int(words[5])
    for p, want5 in ((w / 2.0**32, 1), ((w + 1) / 2.0**32, 0)):
        keep = o64.dropout_keep(n, seed, site, step, p)
        assert keep[5] == want5
        thr = math.floor(p * 2.0**32)
        assert np.array_equal(keep, (words >= thr).astype(np.uint8))
    assert np.all(o64.dropout_keep(n, seed, site, step, 0.0) == 1)


def test_dropout_keep_fraction_and_expectation(o64):
    n = 1 << 20
    for p in (0.1, 0.5):
        keep = o64.dropout_keep(n, 99, 1, 0, p)
        sigma = math.sqrt(p * (1 - p) / n)
        assert abs(keep.mean() - (1 - p)) < 6 * sigma, (p, keep.mean())
        # inverted dropout: the mean of the dropped-out ones stays 1
        y = o64.dropout_apply(np.ones(n), keep, p)
        assert abs(y.mean() - 1.0) < 6 * sigma / (1 - p)
        assert set(np.unique(y)) <= {0.0, 1.0 / (1.0 - p)}


def test_dropout_seed_site_and_step_each_change_the_mask(o64):
    """Two masks that differ in seed, site or step agree on a fraction
    p^2 + (1-p)^2 of the elements, as independent draws do."""
    n, p = 1 << 18, 0.3
    ref = o64.dropout_keep(n, 5, 4, 2, p)
    expect = p * p + (1 - p) * (1 - p)
    sigma = math.sqrt(expect * (1 - expect) / n)
    for seed, site, step in ((6, 4, 2), (5 + (1 << 32), 4, 2), (5, 5, 2), (5, 4, 3)):
        other = o64.dropout_keep(n, seed, site, step, p)
        agree = (other == ref).mean()
        assert abs(agree - expect) < 6 * sigma, (seed, site, step, agree)
    assert np.array_equal(o64.dropout_keep(n, 5, 4, 2, p), ref)


def test_dropout_p0_equals_no_dropout_exactly(o64):
    params, tok, tgt = tiny_inputs()
    m = o64.model(TINY.dims(), TINY.B, TINY.T)
    loss = m.forward(params, tok, tgt)
    g = m.backward(params)
    md = o64.model(TINY.dims(), TINY.B, TINY.T)
    md.set_dropout(0.0, seed=3)
    assert md.forward(params, tok, tgt) == loss
    assert np.array_equal(md.backward(params), g)
    assert np.all(md.keep("att", 1) == 1)


def _torch_dropout_step(cfg, params, tok, tgt, keeps, p):
    """Second opinion for dropout: the architecture in torch float64 with the
    given keep flags applied where the pages put dropout (embedding output,
    attention weights after the softmax, each c_proj output before its residual
    addition), scaled by 1/(1-p); loss and autograd gradients."""
    import torch
    import torch.nn.functional as F
    shapes = syn.tensor_shapes(cfg)
    ts, off = {}, 0
    for name in syn.TENSOR_NAMES:
        n = int(np.prod(shapes[name]))
        ts[name] = torch.tensor(params[off:off + n].reshape(shapes[name]), dtype=torch.float64,
                                requires_grad=True)
        off += n
    B, T = tok.shape
    Cc, H, V = cfg.C, cfg.H, cfg.V
    hs = Cc // H
    s = 1.0 / (1.0 - p)

    def drop(x, k):
        return x * torch.tensor(k.reshape(x.shape), dtype=torch.float64) * s

    tok_t = torch.tensor(tok, dtype=torch.long)
    x = drop(ts["wte"][tok_t] + ts["wpe"][:T], keeps["emb"])
    causal = torch.ones(T, T, dtype=torch.bool).tril()
    for l in range(cfg.L):
        a = F.layer_norm(x, (Cc,), ts["ln1w"][l], ts["ln1b"][l], eps=1e-5)
        qkv = F.linear(a, ts["qkvw"][l], ts["qkvb"][l])
        q, k, v = (z.view(B, T, H, hs).transpose(1, 2) for z in qkv.split(Cc, dim=-1))
        att = (q @ k.transpose(-2, -1)) / math.sqrt(hs)
        att = torch.softmax(att.masked_fill(~causal, float("-inf")), dim=-1)
        att = drop(att, keeps["att"][l])
        y = (att @ v).transpose(1, 2).reshape(B, T, Cc)
        x = x + drop(F.linear(y, ts["attprojw"][l], ts["attprojb"][l]), keeps["attproj"][l])
        a = F.layer_norm(x, (Cc,), ts["ln2w"][l], ts["ln2b"][l], eps=1e-5)
        hmid = F.gelu(F.linear(a, ts["fcw"][l], ts["fcb"][l]), approximate="tanh")
        x = x + drop(F.linear(hmid, ts["fcprojw"][l], ts["fcprojb"][l]), keeps["fcproj"][l])
    x = F.layer_norm(x, (Cc,), ts["lnfw"], ts["lnfb"], eps=1e-5)
    loss = F.cross_entropy((x @ ts["wte"].T).reshape(-1, V), torch.tensor(tgt, dtype=torch.long).reshape(-1))
    loss.backward()
    grads = np.concatenate([ts[k].grad.detach().numpy().reshape(-1) for k in syn.TENSOR_NAMES])
    return float(loss.detach()), grads


@pytest.mark.parametrize("cfg", [
    TINY,
    syn.Config("ragged", V=97, maxT=24, L=3, H=6, C=48, B=3, T=19, lr=3e-3, wd=0.1),
])
def test_dropout_step_matches_torch_autograd(o64, cfg):
    params = syn.init_params(cfg).astype(np.float64)
    tok, tgt = syn.draw_tokens(cfg)
    p = 0.25
    m = o64.model(cfg.dims(), cfg.B, cfg.T)
    m.set_dropout(p, seed=2024, step=1)
    loss = m.forward(params, tok, tgt)
    g = m.backward(params)
    keeps = {"emb": m.keep("emb"),
             "att": [m.keep("att", l) for l in range(cfg.L)],
             "attproj": [m.keep("attproj", l) for l in range(cfg.L)],
             "fcproj": [m.keep("fcproj", l) for l in range(cfg.L)]}
    # the masks are the oracle's definition at each site (site numbering 0, 1 + 3l, ...)
    N = cfg.B * cfg.T
    assert np.array_equal(keeps["emb"], o64.dropout_keep(N * cfg.C, 2024, 0, 1, p))
    assert np.array_equal(keeps["att"][1], o64.dropout_keep(cfg.B * cfg.H * cfg.T ** 2, 2024, 4, 1, p))
    assert np.array_equal(keeps["fcproj"][0], o64.dropout_keep(N * cfg.C, 2024, 3, 1, p))
    t_loss, t_grads = _torch_dropout_step(cfg, params, tok, tgt, keeps, p)
    assert abs(loss - t_loss) < 1e-12
    assert np.abs(g - t_grads).max() < 1e-12 * max(1.0, np.abs(t_grads).max())
    # dropout changed the loss (the masks are in effect)
    m0 = o64.model(cfg.dims(), cfg.B, cfg.T)
    assert abs(m0.forward(params, tok, tgt) - loss) > 1e-6


def test_dropout_gradcheck_directional(o64):
    """With the masks fixed by (seed, step), the dropout loss is a smooth
    function of the parameters: central differences match the backward."""
    params, tok, tgt = tiny_inputs()
    m = o64.model(TINY.dims(), TINY.B, TINY.T)
    m.set_dropout(0.4, seed=77, step=5)
    m.forward(params, tok, tgt)
    grads = m.backward(params)
    rng = np.random.default_rng(16)
    for _ in range(2):
        d = rng.normal(size=params.size)
        h = 1e-6
        f = lambda s: m.forward(params + s * h * d, tok, tgt)
        fd = (-f(2) + 8 * f(1) - 8 * f(-1) + f(-2)) / (12 * h)
        assert abs(fd - grads @ d) <= 1e-6 * abs(grads @ d) + 1e-9
