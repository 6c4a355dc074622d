"""Dropout through the C ABI against the oracle: the keep bits (bit-exact with
the oracle's Philox4x32-10 draws), the element-wise dropout kernels, attention
with dropout on its weights in every kernel family, and the whole training step
with dropout at the four sites; plus the call rules (evaluation without
dropout, p = 0 gives the step without dropout, a fresh mask every forward)."""
import numpy as np
import pytest

from gpt_decoder_step_train_b300 import synthetic as syn
from gpu_util import TOL, per_tensor, rel_l2

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

_keep = []


@pytest.fixture(autouse=True)
def _release():
    yield
    torch.cuda.synchronize()
    _keep.clear()


@pytest.fixture(scope="module")
def B_():
    from gpt_decoder_step_train_b300 import binding
    binding.lib()
    return binding


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    t = t.to(dtype).cuda() if dtype is not None else t.cuda()
    _keep.append(t)
    return t


def host(t):
    torch.cuda.synchronize()
    return t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()


def pack_bits(keep, rows, cols):
    """Oracle keep flags [rows * cols] -> the library's row-wise words."""
    W = (cols + 31) // 32
    k = np.zeros((rows, W * 32), dtype=np.uint64)
    k[:, :cols] = keep.reshape(rows, cols)
    k = k.reshape(rows, W, 32)
    return (k << np.arange(32, dtype=np.uint64)).sum(-1).astype(np.uint32)


def gpu_mask(B_, rows, cols, causal_T, seed, site, step, p):
    L = B_.lib()
    words = L.gpt2_op_dropout_mask_words(rows, cols)
    bits = torch.full((max(words, 1),), 0xA5A5A5A5 - (1 << 32), dtype=torch.int32, device="cuda")
    assert L.gpt2_op_dropout_mask(B_.ptr(bits), rows, cols, causal_T, seed, site, step, p, None) == 0
    return bits


# causal rows with cols % 4 == 0 take the transposed kernel: T = 64; T = 100 (32-row
# groups straddle (batch, head) boundaries); T = 1100 (more than 32 words per row)
@pytest.mark.parametrize("rows,cols,causal_T", [(37, 100, 0), (1, 3, 0), (2 * 3 * 77, 77, 77), (4 * 64, 64, 64),
                                                (2 * 3 * 100, 100, 100), (1100, 1100, 1100)])
@pytest.mark.parametrize("p", [0.0, 0.1, 0.5])
def test_mask_bits_equal_the_oracle_draws(B_, o64, rows, cols, causal_T, p):
    seed, site, step = 0xDEADBEEF12345678, 5, 3
    bits = host(gpu_mask(B_, rows, cols, causal_T, seed, site, step, p)).view(np.uint32)
    want = pack_bits(o64.dropout_keep(rows * cols, seed, site, step, p), rows, cols)
    got = bits[:want.size].reshape(want.shape)
    if causal_T:
        # words past the diagonal are written as 0 and never read
        i = np.arange(rows) % causal_T
        live = (32 * np.arange(want.shape[1]))[None, :] <= i[:, None]
        assert np.all(got[~live] == 0)
        want = np.where(live, want, 0)
    assert np.array_equal(got, want)


def test_mask_bits_full_size_attention_rows(B_, o64):
    """The attention-weight site at the full training shape (B=16, H=12,
    T=1024): every drawn word equals the oracle's, checked on sampled rows."""
    B, H, T = 16, 12, 1024
    rows, seed, site, step, p = B * H * T, 99, 1 + 3 * 11, 7, 0.1
    bits = host(gpu_mask(B_, rows, T, T, seed, site, step, p)).view(np.uint32).reshape(rows, T // 32)
    keep = o64.dropout_keep(rows * T, seed, site, step, p)
    rng = np.random.default_rng(3)
    sample = np.concatenate([[0, T - 1, rows - 1], rng.integers(0, rows, 300)])
    want = pack_bits(keep.reshape(rows, T)[sample].reshape(-1), len(sample), T)
    i = sample % T
    live = (32 * np.arange(T // 32))[None, :] <= i[:, None]
    assert np.array_equal(np.where(live, bits[sample], 0), np.where(live, want, 0))
    kept = keep.reshape(rows, T)[sample]
    assert abs(kept.mean() - 0.9) < 0.01


def test_dropout_residual_and_backward_match_oracle(B_, o64):
    L = B_.lib()
    N, C, p, seed = 37, 100, 0.3, 11
    rng = np.random.default_rng(1)
    out = rng.normal(size=(N, C)).astype(np.float32)
    res = rng.normal(size=(N, C)).astype(np.float32)
    bits = gpu_mask(B_, N, C, 0, seed, 2, 0, p)
    keep = o64.dropout_keep(N * C, seed, 2, 0, p).reshape(N, C)
    for with_res in (True, False):
        o = dev(out)
        r = dev(res) if with_res else None
        assert L.gpt2_op_dropout_residual(B_.ptr(o), B_.ptr(r) if r is not None else None, B_.ptr(bits), N, C, p,
                                          None) == 0
        want = o64.dropout_apply(out, keep, p) + (res if with_res else 0.0)
        assert np.abs(host(o) - want).max() <= 1e-6 * np.abs(want).max()
    g = dev(out)
    d32 = torch.empty(N, C, device="cuda")
    d16 = torch.empty(N, C, dtype=torch.bfloat16, device="cuda")
    assert L.gpt2_op_dropout_backward(B_.ptr(d32), 0, B_.ptr(g), B_.ptr(bits), N, C, p, None) == 0
    assert L.gpt2_op_dropout_backward(B_.ptr(d16), 1, B_.ptr(g), B_.ptr(bits), N, C, p, None) == 0
    want = o64.dropout_apply(out, keep, p)
    assert np.abs(host(d32) - want).max() <= 1e-6 * np.abs(want).max()
    assert np.abs(host(d16) - want).max() <= 2.0 ** -8 * np.abs(want).max()
    assert np.array_equal(host(d16) == 0, keep == 0)
    # in place, fp32
    assert L.gpt2_op_dropout_backward(B_.ptr(g), 0, B_.ptr(g), B_.ptr(bits), N, C, p, None) == 0
    assert np.array_equal(host(g), host(d32))
    # argument checks
    assert L.gpt2_op_dropout_residual(B_.ptr(d32), None, B_.ptr(bits), N, C, 1.0, None) == B_.GPT2_EINVAL
    assert L.gpt2_op_dropout_backward(B_.ptr(d32), 0, B_.ptr(g), B_.ptr(bits), N, 6, p, None) == B_.GPT2_EINVAL
    assert L.gpt2_op_dropout_mask(B_.ptr(bits), 10, 7, 7, 1, 1, 0, 0.1, None) == B_.GPT2_EINVAL  # rows % T
    assert L.gpt2_op_dropout_mask(B_.ptr(bits), 10, 5, 0, 1, 1, 0, -0.1, None) == B_.GPT2_EINVAL


@pytest.mark.parametrize("N,C", [(300, 768), (37, 100)])
@pytest.mark.parametrize("bf16", [False, True])
def test_layernorm_backward_feeding_a_dropped_branch(B_, o64, N, C, bf16):
    """The LayerNorm backward that also writes the dropped branch's gradient
    keep o dx / (1 - p) and its column sum, against the oracle's LayerNorm
    backward followed by its dropout."""
    L = B_.lib()
    p, seed = 0.25, 42
    rng = np.random.default_rng(8)
    x = rng.normal(size=(N, C)).astype(np.float32)
    w = rng.normal(size=C).astype(np.float32)
    b = rng.normal(size=C).astype(np.float32)
    dy = rng.normal(size=(N, C)).astype(np.float32)
    dx0 = rng.normal(size=(N, C)).astype(np.float32)
    _, wm, wr = o64.layernorm_forward(x, w, b)
    bits = gpu_mask(B_, N, C, 0, seed, 6, 1, p)
    keep = o64.dropout_keep(N * C, seed, 6, 1, p).reshape(N, C)
    dx = dev(dx0.copy())
    dxd = torch.empty(N, C, dtype=torch.bfloat16 if bf16 else torch.float32, device="cuda")
    dw, db, ds = (torch.empty(C, device="cuda") for _ in range(3))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    nb = L.gpt2_op_layernorm_backward_scratch_bytes(N, C)
    sc = torch.empty(nb, dtype=torch.uint8, device="cuda")
    assert L.gpt2_op_layernorm_backward_dropout(
        B_.ptr(dx), B_.ptr(dxd), int(bf16), B_.ptr(dw), B_.ptr(db), B_.ptr(ds), B_.ptr(dev(dy)), B_.ptr(dev(x)),
        B_.ptr(dev(w)), B_.ptr(dev(wm.astype(np.float32))), B_.ptr(dev(wr.astype(np.float32))), N, C, 1,
        B_.ptr(bits), p, B_.ptr(sc), nb, B_.ptr(st), None) == 0
    wdx, wdw, wdb = o64.layernorm_backward(dy, x, w, wm.astype(np.float32), wr.astype(np.float32))
    want = dx0 + wdx
    want_d = o64.dropout_apply(want, keep, p)
    assert rel_l2(host(dx), want) < 1e-6
    assert rel_l2(host(dw), wdw) < 1e-6 and rel_l2(host(db), wdb) < 1e-6
    assert rel_l2(host(dxd), want_d) < (4e-3 if bf16 else 1e-6)
    assert np.array_equal(host(dxd) == 0, keep == 0)
    assert rel_l2(host(ds), want_d.sum(axis=0)) < 1e-5
    assert int(st.item()) == 0
    if C > 768 or bf16:
        return
    big = 1024
    assert L.gpt2_op_layernorm_backward_dropout(
        B_.ptr(dx), B_.ptr(dxd), 0, B_.ptr(dw), B_.ptr(db), B_.ptr(ds), B_.ptr(dev(dy)), B_.ptr(dev(x)),
        B_.ptr(dev(w)), B_.ptr(dev(wm.astype(np.float32))), B_.ptr(dev(wr.astype(np.float32))), 1, big, 1,
        B_.ptr(bits), p, B_.ptr(sc), nb, B_.ptr(st), None) in (B_.GPT2_ENOTSUP, B_.GPT2_ENOMEM)


# mode, B, T, C, H: the CUDA-core kernels (fp32; tf32, which takes them under
# dropout; bf16 with head sizes other than 64) and the tcgen05 kernels (bf16, hs 64)
ATT_CASES = [
    ("fp32", 2, 77, 48, 3),
    ("fp32", 1, 200, 128, 2),
    ("tf32", 2, 100, 64, 2),
    ("bf16", 2, 77, 48, 3),
    ("bf16", 2, 200, 128, 2),
    ("bf16", 1, 1024, 128, 2),
    ("bf16", 3, 65, 192, 3),
]


@pytest.mark.parametrize("mode,B,T,C,H", ATT_CASES)
def test_attention_with_dropout_matches_oracle(B_, o64, mode, B, T, C, H):
    L = B_.lib()
    p, seed, site, step = 0.2, 1234, 4, 2
    rng = np.random.default_rng(9)
    qkv = rng.normal(size=(B, T, 3 * C))
    dy = rng.normal(size=(B, T, C))
    bf = mode == "bf16"
    dt = torch.bfloat16 if bf else torch.float32
    if bf:      # the oracle sees the bf16-rounded inputs
        qkv = torch.from_numpy(qkv.astype(np.float32)).to(dt).double().numpy()
        dy = torch.from_numpy(dy.astype(np.float32)).to(dt).double().numpy()
    m = B_.MODES[mode]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bits = gpu_mask(B_, B * H * T, T, T, seed, site, step, p)
    keep = o64.dropout_keep(B * H * T * T, seed, site, step, p)
    q = dev(qkv.astype(np.float32), dt)
    y = torch.empty(B, T, C, dtype=dt, device="cuda")
    lse = torch.empty(B, H, T, device="cuda")
    assert L.gpt2_op_attention_forward_dropout(B_.ptr(y), B_.ptr(lse), B_.ptr(q), B, T, C, H, m, B_.ptr(bits), p,
                                               B_.ptr(st), None) == 0
    wy, P = o64.attention_forward(qkv, H, keep=keep, p=p)
    bar = TOL[mode]["rel"] if mode != "fp32" else 1e-5
    assert rel_l2(host(y), wy) < bar
    # the softmax normaliser is that of the undropped weights
    w0, _ = o64.attention_forward(qkv, H)
    assert rel_l2(wy, w0) > 0.05
    nb = L.gpt2_op_attention_backward_scratch_bytes(B, T, H)
    sc = torch.empty(nb, dtype=torch.uint8, device="cuda")
    dq = torch.full((B, T, 3 * C), 3.0, dtype=dt, device="cuda")
    assert L.gpt2_op_attention_backward_dropout(B_.ptr(dq), B_.ptr(dev(dy.astype(np.float32), dt)), B_.ptr(q),
                                                B_.ptr(y), B_.ptr(lse), B, T, C, H, B_.ptr(sc), nb, m, B_.ptr(bits),
                                                p, B_.ptr(st), None) == 0
    want = o64.attention_backward(dy, qkv, P, H, keep=keep, p=p)
    got = host(dq)
    for i, name in enumerate("qkv"):
        assert rel_l2(got[..., i * C:(i + 1) * C], want[..., i * C:(i + 1) * C]) < bar, name
    assert int(st.item()) == 0
    assert L.gpt2_op_attention_forward_dropout(B_.ptr(y), B_.ptr(lse), B_.ptr(q), B, T, C, H, m, None, p,
                                               B_.ptr(st), None) == B_.GPT2_EINVAL


# ---------------------------------------------------------------- whole step
STEP_CASES = {
    "tiny-fp32": (syn.CONFIGS["tiny"], "fp32"),
    "tiny-bf16": (syn.CONFIGS["tiny"], "bf16"),
    "ragged-tf32": (syn.Config("ragged", V=97, maxT=24, L=3, H=6, C=48, B=3, T=19, lr=1e-4, wd=0.1), "tf32"),
    "124M_small-bf16": (syn.CONFIGS["124M_small"], "bf16"),
}


@pytest.mark.parametrize("name", list(STEP_CASES))
def test_step_with_dropout_matches_oracle(B_, o64, name):
    """Three training forwards under one seed (forward calls 0, 1, 2: drawn
    directly, captured into a graph, replayed) each match the oracle's loss
    with that call's masks; the backward of the last matches per tensor."""
    from gpt_decoder_step_train_b300.binding import GPT2
    cfg, mode = STEP_CASES[name]
    p, seed = 0.1, 20240607
    params = syn.init_params(cfg, perturbed=True)
    tok, tgt = syn.draw_tokens(cfg)
    B, T = tok.shape
    tp = torch.from_numpy(params.copy()).cuda()
    model = GPT2(cfg, tp, maxB=B, mode=mode)
    assert model.set_dropout(p, seed) == 0
    t_tok, t_tgt = torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda()
    om = o64.model(cfg.dims(), B, T)
    p64 = params.astype(np.float64)
    tol = TOL[mode]
    for n in range(3):
        loss = model.forward(t_tok, t_tgt)
        assert model.status() == 0
        om.set_dropout(p, seed=seed, step=n)
        want = om.forward(p64, tok, tgt)
        assert abs(loss - want) <= tol["loss"], (n, loss, want)
    assert model.backward() == 0
    g = model.grads().cpu().numpy().copy()
    og = om.backward(p64)
    gt, ot = per_tensor(cfg, g), per_tensor(cfg, og)
    errs = {k: rel_l2(gt[k], ot[k]) for k in gt}
    assert max(errs.values()) <= tol["rel"], sorted(errs.items(), key=lambda kv: -kv[1])[:4]
    # the masks are in effect: the gradients without dropout are far from these
    om.set_dropout(-1)
    om.forward(p64, tok, tgt)
    assert rel_l2(om.backward(p64), og) > 10 * tol["rel"]
    model.close()


def test_p0_gives_the_step_without_dropout_and_eval_ignores_dropout(B_):
    from gpt_decoder_step_train_b300.binding import GPT2
    cfg = syn.CONFIGS["tiny"]
    params = syn.init_params(cfg, perturbed=True)
    tok, tgt = syn.draw_tokens(cfg)
    t_tok, t_tgt = torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda()
    for mode in ("fp32", "bf16"):
        model = GPT2(cfg, torch.from_numpy(params.copy()).cuda(), maxB=tok.shape[0], mode=mode)
        runs = []
        for p in (0.0, 0.3, 0.0):
            assert model.set_dropout(p, 5) == 0
            ev = model.eval(t_tok, t_tgt)
            losses = [model.forward(t_tok, t_tgt) for _ in range(3)]      # direct, capture, replay
            assert model.backward() == 0
            runs.append((ev, losses, model.grads().cpu().numpy().copy()))
        (e0, l0, g0), (e1, l1, g1), (e2, l2, g2) = runs
        assert e0 == e1 == e2                      # evaluation never drops
        assert l0[0] == l0[1] == l0[2] == l2[0] == l2[2] and np.array_equal(g0, g2)
        assert len(set(l1)) == 3 and abs(l1[0] - l0[0]) > 1e-4   # a new mask every forward
        model.close()


def test_set_dropout_rules(B_):
    from gpt_decoder_step_train_b300.binding import GPT2
    cfg = syn.CONFIGS["tiny"]
    model = GPT2(cfg, torch.from_numpy(syn.init_params(cfg)).cuda(), mode="fp32")
    tok, tgt = syn.draw_tokens(cfg)
    assert model.set_dropout(1.0, 0) == B_.GPT2_EINVAL
    assert model.status() == B_.GPT2_EINVAL
    assert model.set_dropout(-0.5, 0) == B_.GPT2_EINVAL
    model.status()
    assert np.isfinite(model.forward(torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda()))
    assert model.set_dropout(0.2, 1) == 0
    assert model.backward() == B_.GPT2_ESTATE        # the forward was under other settings
    model.status()
    assert np.isfinite(model.forward(torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda()))
    assert model.backward() == 0
    assert model.status() == 0
    model.close()


def test_fullsize_dropout_row0_matches_oracle(B_, o64):
    """The training forward of the GPT-2 124M B16 T1024 workload in bf16 mode
    with dropout p = 0.1 at all four sites: row 0's losses equal a one-row
    oracle forward under the same seed and step (element e of every site has
    the same index in a one-row run for row 0: (0 T + t) C + c, and
    ((0 H + h) T + i) T + j for the attention weights), and the masks matter
    (the GPU row is nearer the dropped oracle row than the undropped one)."""
    from gpt_decoder_step_train_b300.binding import GPT2
    cfg = syn.CONFIGS["124M"]
    p, seed = 0.1, 777
    params = syn.init_params(cfg)
    tok, tgt = syn.draw_tokens(cfg)
    tp = torch.from_numpy(params.copy()).cuda()
    model = GPT2(cfg, tp, maxB=cfg.B, mode="bf16")
    assert model.set_dropout(p, seed) == 0
    loss = model.forward(torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda())
    assert model.status() == 0 and np.isfinite(loss)
    g_row = model.losses(cfg.B * cfg.T).cpu().numpy().reshape(cfg.B, cfg.T)[0].astype(np.float64)
    model.close()
    om = o64.model(cfg.dims(), 1, cfg.T)
    p64 = params.astype(np.float64)
    om.set_dropout(p, seed=seed, step=0)
    o_mean = om.forward(p64, tok[:1], tgt[:1])
    o_row = om.losses().astype(np.float64)
    assert abs(g_row.mean() - o_mean) <= TOL["bf16"]["loss"], (g_row.mean(), o_mean)
    assert rel_l2(g_row, o_row) <= TOL["bf16"]["rel"]
    # the masks matter: the row is nearer the dropped oracle row than the undropped one
    om.set_dropout(-1)
    om.forward(p64, tok[:1], tgt[:1])
    assert rel_l2(g_row, o_row) < rel_l2(g_row, om.losses().astype(np.float64))
