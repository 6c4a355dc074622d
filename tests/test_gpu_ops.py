"""Per-kernel parity: each C-ABI op on the GPU against the oracle's layer
function on the same seeded inputs, at shapes that span several tiles and
leave ragged tails."""
import math

import numpy as np
import pytest

from gpu_util import rel_l2

from gpt_decoder_step_train_b300 import synthetic as syn

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

MODES = ["fp32", "tf32"]


@pytest.fixture(scope="module")
def L():
    from gpt_decoder_step_train_b300 import binding
    return binding.lib()


@pytest.fixture(scope="module")
def B_():
    from gpt_decoder_step_train_b300 import binding
    return binding


_keep = []     # device copies stay alive until the test ends (kernels run asynchronously)
_status = []   # device status word shared by the GEMM / attention calls of one test


@pytest.fixture(autouse=True)
def _release_device_copies():
    _status.append(torch.zeros(1, dtype=torch.int32, device="cuda"))
    yield
    torch.cuda.synchronize()
    st = int(_status.pop().cpu()[0])
    _keep.clear()
    assert st == 0, f"device status {st} (a bounded wait timed out)"


def S():
    from gpt_decoder_step_train_b300 import binding
    return binding.ptr(_status[-1])


def dev(a):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    _keep.append(t)
    return t


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def tol(mode, strict=1e-5, tc=5e-3):
    return strict if mode == "fp32" else tc


# ------------------------------------------------------------------ encoder

def test_encoder_forward_bit_exact(L, B_, o32):
    rng = np.random.default_rng(0)
    V, maxT, C, B, T = 1000, 300, 96, 3, 257
    wte = rng.normal(size=(V, C)).astype(np.float32)
    wpe = rng.normal(size=(maxT, C)).astype(np.float32)
    tok = rng.integers(0, V, (B, T)).astype(np.int32)
    x = torch.empty(B * T, C, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = L.gpt2_op_encoder_forward(B_.ptr(x), B_.ptr(dev(tok)), B_.ptr(dev(wte)), B_.ptr(dev(wpe)),
                                   B, T, C, V, B_.ptr(st), None)
    assert rc == 0
    want = o32.encoder_forward(tok, wte, wpe).reshape(B * T, C)
    assert np.array_equal(host(x), want)
    assert int(host(st)[0]) == 0


def test_encoder_forward_flags_bad_token(L, B_):
    V, C, B, T = 50, 8, 1, 4
    tok = np.array([[1, 2, 50, -1]], dtype=np.int32)
    x = torch.empty(B * T, C, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    wte = torch.ones(V, C, device="cuda")
    wpe = torch.ones(8, C, device="cuda")
    assert L.gpt2_op_encoder_forward(B_.ptr(x), B_.ptr(dev(tok)), B_.ptr(wte), B_.ptr(wpe), B, T, C,
                                     V, B_.ptr(st), None) == 0
    assert int(host(st)[0]) & B_.STATUS_BAD_TOKEN
    assert np.all(host(x)[2:] == 0)


@pytest.mark.parametrize("kind", ["uniform", "zipf", "one_id", "zipf_full"])
def test_encoder_backward_matches_and_is_deterministic(L, B_, o64, kind):
    rng = np.random.default_rng(1)
    V, maxT, C, B, T = 5000, 200, 64, 4, 199
    if kind == "zipf":         # heavy repetition of a few ids, like the training token stream
        tok = np.minimum(rng.zipf(1.3, (B, T)) - 1, V - 1).astype(np.int32)
    elif kind == "one_id":     # one bucket of 2048 entries: the shared-memory sort of large buckets
        V, maxT, B, T = 50, 1024, 2, 1024
        tok = np.full((B, T), 7, dtype=np.int32)
    elif kind == "zipf_full":  # the GPT-2 124M B16 T1024 shape: several buckets above 256 entries
        V, maxT, C, B, T = 50257, 1024, 768, 16, 1024
        tok = syn.draw_tokens(syn.CONFIGS["124M"])[0]
    else:
        tok = rng.integers(0, V, (B, T)).astype(np.int32)
    dx = rng.normal(size=(B * T, C)).astype(np.float32)
    base = rng.normal(size=(V, C)).astype(np.float32)   # dwte already holds the lm_head part
    nbytes = L.gpt2_op_encoder_backward_scratch_bytes(B * T, V, C)
    outs = []
    for _ in range(2):
        dwte = dev(base.copy())
        dwpe = torch.full((maxT, C), 7.0, device="cuda")
        scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        rc = L.gpt2_op_encoder_backward(B_.ptr(dwte), B_.ptr(dwpe), B_.ptr(dev(dx)),
                                        B_.ptr(dev(tok)), B, T, maxT, C, V, B_.ptr(scratch),
                                        nbytes, None)
        assert rc == 0
        outs.append((host(dwte), host(dwpe)))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    w_dwte, w_dwpe = o64.encoder_backward(dx.reshape(B, T, C), tok, V, maxT)
    assert rel_l2(outs[0][0] - base, w_dwte) < 1e-6
    assert rel_l2(outs[0][1], w_dwpe) < 1e-6
    assert np.all(outs[0][1][T:] == 0)


def test_encoder_backward_sizes_up_down_up(L, B_, o64):
    """The same process runs the encoder backward on 16 x 1024 positions, then
    1 x 1024, then 16 x 1024 again (the bitmap kernel's shared memory shrinks
    and grows back), each against the oracle: a kernel's shared-memory limit
    must never be left below a size that an earlier call already set up."""
    V, maxT, C = 50257, 1024, 768
    tok_full = syn.draw_tokens(syn.CONFIGS["124M"])[0]
    rng = np.random.default_rng(3)
    for B in (16, 1, 16):
        tok = np.ascontiguousarray(tok_full[:B])
        T = tok.shape[1]
        dx = rng.normal(size=(B * T, C)).astype(np.float32)
        nbytes = L.gpt2_op_encoder_backward_scratch_bytes(B * T, V, C)
        dwte = torch.zeros(V, C, device="cuda")
        dwpe = torch.zeros(maxT, C, device="cuda")
        scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        rc = L.gpt2_op_encoder_backward(B_.ptr(dwte), B_.ptr(dwpe), B_.ptr(dev(dx)), B_.ptr(dev(tok)), B, T,
                                        maxT, C, V, B_.ptr(scratch), nbytes, None)
        assert rc == 0
        w_dwte, w_dwpe = o64.encoder_backward(dx.reshape(B, T, C), tok, V, maxT)
        assert rel_l2(host(dwte), w_dwte) < 1e-6
        assert rel_l2(host(dwpe), w_dwpe) < 1e-6


# ------------------------------------------------------------------ layernorm

@pytest.mark.parametrize("N,C", [(1000, 768), (37, 64), (513, 1600), (5, 4)])
def test_layernorm_forward(L, B_, o64, N, C):
    rng = np.random.default_rng(2)
    x = (rng.normal(size=(N, C)) * 2 + 0.5).astype(np.float32)
    w = rng.normal(size=C).astype(np.float32)
    b = rng.normal(size=C).astype(np.float32)
    y = torch.empty(N, C, device="cuda")
    mean = torch.empty(N, device="cuda")
    rstd = torch.empty(N, device="cuda")
    assert L.gpt2_op_layernorm_forward(B_.ptr(y), B_.ptr(mean), B_.ptr(rstd), B_.ptr(dev(x)),
                                       B_.ptr(dev(w)), B_.ptr(dev(b)), N, C, None) == 0
    wy, wm, wr = o64.layernorm_forward(x, w, b)
    assert rel_l2(host(y), wy) < 1e-6
    assert rel_l2(host(mean), wm) < 1e-6
    assert rel_l2(host(rstd), wr) < 1e-6


@pytest.mark.parametrize("accumulate", [1, 0])
@pytest.mark.parametrize("N,C", [(1000, 768), (37, 64), (513, 1600), (16384, 768), (3, 2048), (300, 1024), (4096, 1600)])
def test_layernorm_backward(L, B_, o64, N, C, accumulate):
    rng = np.random.default_rng(3)
    x = rng.normal(size=(N, C)).astype(np.float32)
    w = rng.normal(size=C).astype(np.float32)
    b = rng.normal(size=C).astype(np.float32)
    dy = rng.normal(size=(N, C)).astype(np.float32)
    dx0 = rng.normal(size=(N, C)).astype(np.float32)    # residual gradient accumulated into
    _, wm, wr = o64.layernorm_forward(x, w, b)
    mean, rstd = dev(wm.astype(np.float32)), dev(wr.astype(np.float32))
    dx = dev(dx0.copy() if accumulate else np.full((N, C), np.nan, np.float32))
    dw = torch.empty(C, device="cuda")
    db = torch.empty(C, device="cuda")
    ds = torch.empty(C, device="cuda")
    st = dev(np.zeros(1, np.int32))
    nbytes = L.gpt2_op_layernorm_backward_scratch_bytes(N, C)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    assert L.gpt2_op_layernorm_backward(B_.ptr(dx), None, B_.ptr(dw), B_.ptr(db), B_.ptr(ds), B_.ptr(dev(dy)),
                                        B_.ptr(dev(x)), B_.ptr(dev(w)), B_.ptr(mean), B_.ptr(rstd),
                                        N, C, accumulate, B_.ptr(scratch), nbytes, B_.ptr(st), None) == 0
    wdx, wdw, wdb = o64.layernorm_backward(dy, x, w, wm.astype(np.float32), wr.astype(np.float32))
    want = dx0 + wdx if accumulate else wdx
    assert int(host(st)[0]) == 0
    assert rel_l2(host(dx), want) < 1e-6
    assert rel_l2(host(dw), wdw) < 1e-6
    assert rel_l2(host(db), wdb) < 1e-6
    # the column sum of the resulting gradient (a bias gradient), summed in float64 here
    assert rel_l2(host(ds), want.astype(np.float64).sum(axis=0)) < 1e-5


# ------------------------------------------------------------------ linear

LIN_SHAPES = [(300, 64, 192), (257, 768, 2304), (129, 3072, 768), (128, 64, 65), (64, 768, 50257)]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("N,IC,OC", LIN_SHAPES)
def test_linear_forward_epilogues(L, B_, o64, mode, N, IC, OC):
    rng = np.random.default_rng(4)
    x = rng.normal(size=(N, IC)).astype(np.float32)
    w = (rng.normal(size=(OC, IC)) * 0.05).astype(np.float32)
    b = rng.normal(size=OC).astype(np.float32)
    res = rng.normal(size=(N, OC)).astype(np.float32)
    ref = o64.matmul_forward(x, w, b)
    m = B_.MODES[mode]
    # plain + bias, padded output stride with zero fill
    ld = ((OC + 127) // 128) * 128
    out = torch.full((N, ld), 5.0, device="cuda")
    rc = L.gpt2_op_linear_forward(B_.ptr(out), None, B_.ptr(dev(x)), B_.ptr(dev(w)), B_.ptr(dev(b)),
                                  None, N, IC, OC, ld, B_.GPT2_LINEAR_ZERO_PAD, m, S(), None)
    assert rc == 0
    o = host(out)
    assert rel_l2(o[:, :OC], ref) < tol(mode)
    assert np.all(o[:, OC:] == 0)
    if OC > 4096:
        return
    # residual
    out = dev(res.copy())
    assert L.gpt2_op_linear_forward(B_.ptr(out), None, B_.ptr(dev(x)), B_.ptr(dev(w)),
                                    B_.ptr(dev(b)), B_.ptr(out), N, IC, OC, OC, 0, m, S(), None) == 0
    assert rel_l2(host(out), ref + res) < tol(mode)
    # GELU, keeping the pre-activation
    out = torch.empty(N, OC, device="cuda")
    pre = torch.empty(N, OC, device="cuda")
    assert L.gpt2_op_linear_forward(B_.ptr(out), B_.ptr(pre), B_.ptr(dev(x)), B_.ptr(dev(w)),
                                    B_.ptr(dev(b)), None, N, IC, OC, OC, B_.GPT2_LINEAR_GELU, m,
                                    S(), None) == 0
    assert rel_l2(host(pre), ref) < tol(mode)
    assert rel_l2(host(out), o64.gelu_forward(ref)) < tol(mode)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("N,IC,OC", LIN_SHAPES)
def test_linear_backward(L, B_, o64, mode, N, IC, OC):
    rng = np.random.default_rng(5)
    x = rng.normal(size=(N, IC)).astype(np.float32)
    w = (rng.normal(size=(OC, IC)) * 0.05).astype(np.float32)
    ld = ((OC + 127) // 128) * 128 if OC > 4096 else OC
    dy = np.zeros((N, ld), dtype=np.float32)
    dy[:, :OC] = rng.normal(size=(N, OC))
    m = B_.MODES[mode]
    wdx, wdw, wdb = o64.matmul_backward(dy[:, :OC], x, w)
    dx = torch.empty(N, IC, device="cuda")
    assert L.gpt2_op_linear_backward_input(B_.ptr(dx), B_.ptr(dev(dy)), B_.ptr(dev(w)), None, N, IC,
                                           OC, ld, m, S(), None) == 0
    assert rel_l2(host(dx), wdx) < tol(mode)
    # with the GELU derivative of a pre-activation h
    h = rng.normal(size=(N, IC)).astype(np.float32)
    assert L.gpt2_op_linear_backward_input(B_.ptr(dx), B_.ptr(dev(dy)), B_.ptr(dev(w)),
                                           B_.ptr(dev(h)), N, IC, OC, ld, m, S(), None) == 0
    assert rel_l2(host(dx), o64.gelu_backward(h, wdx)) < tol(mode)
    dw = torch.empty(OC, IC, device="cuda")
    db = torch.empty(OC, device="cuda")
    nbytes = L.gpt2_op_linear_backward_weight_scratch_bytes(N, IC, OC, m)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    assert L.gpt2_op_linear_backward_weight(B_.ptr(dw), B_.ptr(db), B_.ptr(dev(dy)), B_.ptr(dev(x)),
                                            N, IC, OC, ld, B_.ptr(scratch), nbytes, m, S(), None) == 0
    assert rel_l2(host(dw), wdw) < tol(mode)
    assert rel_l2(host(db), wdb) < 1e-6


# ------------------------------------------------------------------ attention

# head size 64 (tcgen05 forward in tf32 mode): T = 300 and 129 (ragged query and
# key tiles; at T = 300 an item's second query tile is empty), T = 1024 (eight
# key tiles, four items per (batch, head)), 300 items of T = 128 (two or three
# items per CTA of the persistent grid)
ATT_SHAPES = [(2, 37, 64, 4), (1, 300, 768, 12), (2, 129, 192, 3), (1, 1, 64, 4), (3, 64, 48, 6),
              (2, 1024, 256, 4), (25, 128, 768, 12)]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("B,T,C,H", ATT_SHAPES)
def test_attention_forward_backward(L, B_, o64, mode, B, T, C, H):
    rng = np.random.default_rng(6)
    qkv = rng.normal(size=(B, T, 3 * C)).astype(np.float32)
    dy = rng.normal(size=(B, T, C)).astype(np.float32)
    m = B_.MODES[mode]
    y = torch.empty(B, T, C, device="cuda")
    lse = torch.empty(B, H, T, device="cuda")
    d_qkv = dev(qkv)
    assert L.gpt2_op_attention_forward(B_.ptr(y), B_.ptr(lse), B_.ptr(d_qkv), B, T, C, H, m,
                                       S(), None) == 0
    wy, P = o64.attention_forward(qkv, H)
    assert rel_l2(host(y), wy) < tol(mode)
    # lse from the oracle's scores: P_ij = exp(s_ij - lse_i) for j <= i
    hs = C // H
    q = qkv[:, :, :C].reshape(B, T, H, hs).transpose(0, 2, 1, 3).astype(np.float64)
    k = qkv[:, :, C:2 * C].reshape(B, T, H, hs).transpose(0, 2, 1, 3).astype(np.float64)
    s = q @ k.transpose(0, 1, 3, 2) / math.sqrt(hs)
    mask = np.tril(np.ones((T, T), dtype=bool))
    s = np.where(mask, s, -np.inf)
    mx = s.max(-1)
    wl = mx + np.log(np.exp(s - mx[..., None]).sum(-1))
    assert np.abs(host(lse) - wl).max() < tol(mode, 1e-5, 2e-2)
    dqkv = torch.full((B, T, 3 * C), 3.0, device="cuda")
    nbytes = L.gpt2_op_attention_backward_scratch_bytes(B, T, H)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    assert L.gpt2_op_attention_backward(B_.ptr(dqkv), B_.ptr(dev(dy)), B_.ptr(d_qkv), B_.ptr(y),
                                        B_.ptr(lse), B, T, C, H, B_.ptr(scratch), nbytes, m,
                                        S(), None) == 0
    want = o64.attention_backward(dy, qkv, P, H)
    got = host(dqkv)
    for i, name in enumerate("qkv"):
        assert rel_l2(got[..., i * C:(i + 1) * C], want[..., i * C:(i + 1) * C]) < tol(mode), name


# ------------------------------------------------------------------ cross-entropy

@pytest.mark.parametrize("N,V", [(37, 65), (64, 50257), (5, 1)])
def test_crossentropy(L, B_, o64, N, V):
    rng = np.random.default_rng(7)
    ld = ((V + 127) // 128) * 128
    z = np.zeros((N, ld), dtype=np.float32)
    z[:, :V] = rng.normal(size=(N, V)) * 3
    z[:, V:] = 1e30          # padding must be ignored
    tgt = rng.integers(0, V, N).astype(np.int32)
    losses = torch.empty(N, device="cuda")
    dz = dev(z)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert L.gpt2_op_crossentropy(B_.ptr(losses), B_.ptr(dz), None, B_.ptr(dev(tgt)), N, V, ld,
                                  1.0 / N, B_.ptr(st), None) == 0
    mean, wl, probs = o64.crossentropy_forward(z, tgt, V=V)
    wdz = o64.crossentropy_backward(probs, tgt, ld=ld)
    assert rel_l2(host(losses), wl) < 1e-6
    g = host(dz)
    assert rel_l2(g, wdz) < 1e-5
    assert np.all(g[:, V:] == 0)
    # target selection is exact: the one negative gradient entry of each row sits at the target
    if V > 1:
        assert np.array_equal(np.argmin(g[:, :V], axis=1), tgt)
        assert np.all((g[:, :V] < 0).sum(1) == 1)
    out = torch.empty(1, device="cuda")
    assert L.gpt2_op_sum(B_.ptr(out), B_.ptr(losses), N, 1.0 / N, None) == 0
    assert abs(float(host(out)[0]) - mean) < 1e-5


def test_crossentropy_flags_bad_target(L, B_):
    N, V, ld = 3, 10, 128
    z = torch.zeros(N, ld, device="cuda")
    tgt = dev(np.array([1, 10, 2], dtype=np.int32))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    losses = torch.empty(N, device="cuda")
    assert L.gpt2_op_crossentropy(B_.ptr(losses), B_.ptr(z), None, B_.ptr(tgt), N, V, ld, 1.0,
                                  B_.ptr(st), None) == 0
    assert int(host(st)[0]) & B_.STATUS_BAD_TARGET
    assert np.all(host(z)[1] == 0) and host(losses)[1] == 0


# ------------------------------------------------------------------ AdamW

def test_adamw(L, B_, o32):
    rng = np.random.default_rng(8)
    n = 100_004
    p = rng.normal(size=n).astype(np.float32)
    g = (rng.normal(size=n) * 1e-2).astype(np.float32)
    m0 = (rng.normal(size=n) * 1e-3).astype(np.float32)
    v0 = np.abs(rng.normal(size=n) * 1e-4).astype(np.float32)
    t, lr, b1, b2, eps, wd = 7, 6e-4, 0.9, 0.999, 1e-8, 0.1
    dp, dm, dv = dev(p), dev(m0), dev(v0)
    bc1, bc2 = 1 - b1 ** t, 1 - b2 ** t
    assert L.gpt2_op_adamw(B_.ptr(dp), B_.ptr(dev(g)), B_.ptr(dm), B_.ptr(dv), n, lr, b1, b2, eps,
                           wd, bc1, bc2, None) == 0
    wp, wm, wv = p.copy(), m0.copy(), v0.copy()
    o32.adamw(wp, g, wm, wv, lr, b1, b2, eps, wd, t)
    assert rel_l2(host(dp), wp) < 1e-7
    assert rel_l2(host(dm), wm) < 1e-6
    assert rel_l2(host(dv), wv) < 1e-6
