"""bf16 operand path: each kernel against the oracle on bf16-rounded inputs.

The oracle computes in float64 on exactly the values the GPU reads (inputs
rounded to bf16 first), so the remaining differences are fp32 accumulation and
the final rounding of bf16 outputs (relative 2^-9 per element).
"""
import ctypes

import numpy as np
import pytest

from gpu_util import rel_l2

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

BF16_OUT = 4e-3          # rel-L2 of a bf16-rounded output (2^-9 per element, rms)
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


def bf(a):
    """bf16 device tensor from a float array (round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).cuda()
    _keep.append(t)
    return t


def f32(a):
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    _keep.append(t)
    return t


def rounded(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def host(t):
    torch.cuda.synchronize()
    return t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()


def test_to_bf16_is_round_to_nearest_even(B_):
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(size=100_003) * 10 ** rng.uniform(-30, 30, 100_003),
                        [0.0, -0.0, 1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -9, 3.4e38, 1e-40]]).astype(np.float32)
    src = f32(x)
    out = torch.empty(x.size, dtype=torch.bfloat16, device="cuda")
    assert B_.lib().gpt2_op_to_bf16(B_.ptr(out), B_.ptr(src), x.size, None) == 0
    want = torch.from_numpy(x).to(torch.bfloat16)
    assert torch.equal(out.cpu().view(torch.int16), want.view(torch.int16))


# shapes of at least 256 x 256 run on CTA pairs (cta_group::2), the others on single CTAs
GEMM_SHAPES = [(300, 192, 64), (257, 2304, 768), (129, 768, 3072), (128, 65, 64), (64, 50304, 768),
               (512, 768, 3072), (1024, 2304, 768), (384, 520, 256), (512, 50304, 768)]


def _gemm(B_, M, N, K, A, lda, ak, Bm, ldb, bk, out, ldo, out_bf16, **epi):
    a = B_.gpt2_gemm_args()
    a.M, a.N, a.K = M, N, K
    a.A, a.lda, a.a_kmajor = A.data_ptr(), lda, ak
    a.B, a.ldb, a.b_kmajor = Bm.data_ptr(), ldb, bk
    a.bf16 = 1
    a.out, a.ldo, a.out_bf16 = out.data_ptr(), ldo, out_bf16
    for k in ("out_pre", "bias", "residual", "gelu_x", "colsum"):
        t = epi.get(k)
        setattr(a, k, t.data_ptr() if t is not None else None)
    a.ldg = epi.get("ldg", 0)
    a.gelu = epi.get("gelu", 0)
    a.pre_bf16 = epi.get("pre_bf16", 0)
    a.gelu_x_bf16 = epi.get("gelu_x_bf16", 0)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = B_.lib().gpt2_op_gemm(ctypes.addressof(a), B_.GPT2_MODE_BF16, B_.ptr(st), None)
    torch.cuda.synchronize()
    assert rc == 0 and int(st.item()) == 0


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_bf16_gemm_three_products(B_, o64, M, N, K):
    rng = np.random.default_rng(1)
    a = rng.normal(size=(M, K))
    b = rng.normal(size=(N, K)) * 0.05
    ar, br = rounded(a), rounded(b)
    want = o64.matmul_forward(ar, br)                      # A B^T
    # outputs use a row stride padded to 16 bytes, as the model's buffers do
    ldo = (N + 7) // 8 * 8
    # forward: A K-major [M,K], B K-major [N,K]
    outp = torch.empty(M, ldo, device="cuda")
    out = outp[:, :N]
    _gemm(B_, M, N, K, bf(a), K, 1, bf(b), K, 1, outp, ldo, 0)
    assert rel_l2(host(out), want) < 1e-5
    if N % 8:
        # a bf16 row of N elements is not 16-byte aligned: TMA cannot read the N-major forms
        a_ = B_.gpt2_gemm_args()
        a_.M, a_.N, a_.K, a_.A, a_.lda, a_.a_kmajor = M, N, K, bf(a).data_ptr(), K, 1
        a_.B, a_.ldb, a_.b_kmajor, a_.bf16 = bf(b.T).data_ptr(), N, 0, 1
        a_.out, a_.ldo = outp.data_ptr(), ldo
        assert B_.lib().gpt2_op_gemm(ctypes.addressof(a_), B_.GPT2_MODE_BF16, None, None) == B_.GPT2_ENOTSUP
        return
    # dX form: B N-major [K,N]
    outp.zero_()
    _gemm(B_, M, N, K, bf(a), K, 1, bf(b.T), N, 0, outp, ldo, 0)
    assert rel_l2(host(out), want) < 1e-5
    # dW form: A M-major [K,M], B N-major [K,N] (rows of M bf16 must be 16-byte aligned)
    if M % 8 == 0:
        outp.zero_()
        _gemm(B_, M, N, K, bf(a.T), M, 0, bf(b.T), N, 0, outp, ldo, 0)
        assert rel_l2(host(out), want) < 1e-5
    if N > 4096:
        return
    # epilogues with bf16 outputs
    bias = rng.normal(size=N)
    res = rng.normal(size=(M, N))
    o16 = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    pre = torch.empty(M, N, device="cuda")
    _gemm(B_, M, N, K, bf(a), K, 1, bf(b), K, 1, o16, N, 1, bias=f32(bias), out_pre=pre, gelu=1)
    assert rel_l2(host(pre), want + bias) < 1e-5
    assert rel_l2(host(o16), o64.gelu_forward(want + bias)) < BF16_OUT
    o32 = torch.empty(M, N, device="cuda")
    _gemm(B_, M, N, K, bf(a), K, 1, bf(b), K, 1, o32, N, 0, bias=f32(bias), residual=f32(res))
    assert rel_l2(host(o32), want + bias + res) < 1e-5
    h = rng.normal(size=(M, N))
    _gemm(B_, M, N, K, bf(a), K, 1, bf(b), K, 1, o16, N, 1, gelu_x=f32(h), ldg=N)
    assert rel_l2(host(o16), o64.gelu_backward(h, want)) < BF16_OUT
    # the step's bf16 forms: pre-activation stored as bf16, GELU input read as bf16,
    # and a plain bias epilogue into bf16
    pre16 = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    _gemm(B_, M, N, K, bf(a), K, 1, bf(b), K, 1, o16, N, 1, bias=f32(bias), out_pre=pre16, gelu=1,
          pre_bf16=1)
    assert rel_l2(host(pre16), want + bias) < BF16_OUT
    assert rel_l2(host(o16), o64.gelu_forward(want + bias)) < BF16_OUT
    groups = (M + 31) // 32
    cs = torch.full((groups, N), 7.0, device="cuda")
    _gemm(B_, M, N, K, bf(a), K, 1, bf(b), K, 1, o16, N, 1, gelu_x=bf(h), ldg=N, gelu_x_bf16=1, colsum=cs)
    dh = o64.gelu_backward(rounded(h), want)
    assert rel_l2(host(o16), dh) < BF16_OUT
    # per-32-row column sums of the unrounded values (the fused bias gradient)
    pad = np.zeros((groups * 32, N))
    pad[:M] = dh
    want_cs = pad.reshape(groups, 32, N).sum(1)
    assert rel_l2(host(cs), want_cs) < BF16_OUT
    assert rel_l2(host(cs).sum(0), dh.sum(0)) < BF16_OUT
    _gemm(B_, M, N, K, bf(a), K, 1, bf(b), K, 1, o16, N, 1, bias=f32(bias))
    assert rel_l2(host(o16), want + bias) < BF16_OUT


@pytest.mark.parametrize("N,C", [(1000, 768), (37, 64), (513, 1600)])
def test_bf16_layernorm(B_, o64, N, C):
    L = B_.lib()
    rng = np.random.default_rng(2)
    x = rng.normal(size=(N, C)) * 2 + 0.5
    w, b = rng.normal(size=C), rng.normal(size=C)
    y16 = torch.empty(N, C, dtype=torch.bfloat16, device="cuda")
    mean, rstd = torch.empty(N, device="cuda"), torch.empty(N, device="cuda")
    assert L.gpt2_op_layernorm_forward_bf16(B_.ptr(y16), B_.ptr(mean), B_.ptr(rstd), B_.ptr(f32(x)),
                                            B_.ptr(f32(w)), B_.ptr(f32(b)), N, C, None) == 0
    wy, wm, wr = o64.layernorm_forward(x.astype(np.float32), w.astype(np.float32), b.astype(np.float32))
    assert rel_l2(host(y16), wy) < BF16_OUT
    assert rel_l2(host(mean), wm) < 1e-6
    # backward: the bf16 copy is the rounded fp32 result
    dy = rng.normal(size=(N, C))
    dx = f32(rng.normal(size=(N, C)))
    dx16 = torch.empty(N, C, dtype=torch.bfloat16, device="cuda")
    dw, db = torch.empty(C, device="cuda"), torch.empty(C, device="cuda")
    nb = L.gpt2_op_layernorm_backward_scratch_bytes(N, C)
    sc = torch.empty(nb, dtype=torch.uint8, device="cuda")
    assert L.gpt2_op_layernorm_backward(B_.ptr(dx), B_.ptr(dx16), B_.ptr(dw), B_.ptr(db), None,
                                        B_.ptr(f32(dy)), B_.ptr(f32(x)), B_.ptr(f32(w)), B_.ptr(mean),
                                        B_.ptr(rstd), N, C, 1, B_.ptr(sc), nb, None, None) == 0
    torch.cuda.synchronize()
    assert torch.equal(dx16.cpu().view(torch.int16), dx.cpu().to(torch.bfloat16).view(torch.int16))


@pytest.mark.parametrize("N,V", [(37, 65), (64, 50257)])
def test_bf16_crossentropy_gradient(B_, o64, N, V):
    L = B_.lib()
    rng = np.random.default_rng(3)
    ld = (V + 127) // 128 * 128
    z = np.zeros((N, ld), dtype=np.float32)
    z[:, :V] = rng.normal(size=(N, V)) * 3
    tgt = rng.integers(0, V, N).astype(np.int32)
    zt = f32(z)
    dz16 = torch.full((N, ld), 7.0, dtype=torch.bfloat16, device="cuda")
    losses = torch.empty(N, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tg = torch.from_numpy(tgt).cuda()
    assert L.gpt2_op_crossentropy(B_.ptr(losses), B_.ptr(zt), B_.ptr(dz16), B_.ptr(tg), N, V, ld, 1.0 / N,
                                  B_.ptr(st), None) == 0
    mean, wl, probs = o64.crossentropy_forward(z, tgt, V=V)
    wdz = o64.crossentropy_backward(probs, tgt, ld=ld)
    g = host(dz16)
    assert np.array_equal(host(zt), z)                     # logits left unchanged
    assert rel_l2(host(losses), wl) < 1e-6
    assert rel_l2(g, wdz) < BF16_OUT
    assert np.all(g[:, V:] == 0)
    assert np.array_equal(np.argmin(g[:, :V], axis=1), tgt)


@pytest.mark.parametrize("N,V", [(37, 65), (300, 50257)])
def test_bf16_logits_crossentropy_in_place(B_, o64, N, V):
    """bf16 logits: losses from the stored bf16 values, gradient written over them."""
    L = B_.lib()
    rng = np.random.default_rng(5)
    ld = (V + 127) // 128 * 128
    z = np.zeros((N, ld), dtype=np.float32)
    z[:, :V] = rng.normal(size=(N, V)) * 3
    z[:, V:] = 9.0                                         # padding garbage: ignored, then zeroed
    tgt = rng.integers(0, V, N).astype(np.int32)
    zt = bf(z)
    losses = torch.empty(N, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tg = torch.from_numpy(tgt).cuda()
    # dscale 0: losses only, logits untouched
    assert L.gpt2_op_crossentropy_bf16(B_.ptr(losses), B_.ptr(zt), B_.ptr(tg), N, V, ld, 0.0,
                                       B_.ptr(st), None) == 0
    zr = rounded(z)
    mean, wl, probs = o64.crossentropy_forward(zr, tgt, V=V)
    assert rel_l2(host(losses), wl) < 1e-6
    assert np.array_equal(host(zt), zr)
    assert L.gpt2_op_crossentropy_bf16(B_.ptr(losses), B_.ptr(zt), B_.ptr(tg), N, V, ld, 1.0 / N,
                                       B_.ptr(st), None) == 0
    wdz = o64.crossentropy_backward(probs, tgt, ld=ld)
    g = host(zt)
    assert rel_l2(host(losses), wl) < 1e-6
    assert rel_l2(g, wdz) < BF16_OUT
    assert np.all(g[:, V:] == 0)
    assert np.array_equal(np.argmin(g[:, :V], axis=1), tgt)   # target selection
    assert int(st.item()) == 0


def test_bf16_logits_crossentropy_flags_bad_target(B_):
    L = B_.lib()
    N, V, ld = 4, 65, 128
    z = bf(np.ones((N, ld)))
    tgt = torch.tensor([0, 65, -1, 64], dtype=torch.int32, device="cuda")
    losses = torch.empty(N, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert L.gpt2_op_crossentropy_bf16(B_.ptr(losses), B_.ptr(z), B_.ptr(tgt), N, V, ld, 1.0,
                                       B_.ptr(st), None) == 0
    lo, g = host(losses), host(z)
    assert int(st.item()) & 2
    assert lo[1] == 0 and lo[2] == 0 and np.all(g[1:3] == 0)
    assert abs(lo[0] - np.log(65)) < 1e-5 and abs(lo[3] - np.log(65)) < 1e-5
    assert L.gpt2_op_crossentropy_bf16(B_.ptr(losses), B_.ptr(z), B_.ptr(tgt), N, V, 8, 1.0,
                                       B_.ptr(st), None) != 0            # ld < V
    assert L.gpt2_op_crossentropy_bf16(B_.ptr(losses), B_.ptr(z), B_.ptr(tgt), N, 60000, 60032, 1.0,
                                       B_.ptr(st), None) != 0            # row above the limit


def test_bf16_bias_grad(B_):
    L = B_.lib()
    rng = np.random.default_rng(4)
    N, OC = 3000, 3072
    d = rng.normal(size=(N, OC))
    db = torch.empty(OC, device="cuda")
    nb = L.gpt2_op_bias_grad_scratch_bytes(N, OC)
    sc = torch.empty(nb, dtype=torch.uint8, device="cuda")
    assert L.gpt2_op_bias_grad(B_.ptr(db), B_.ptr(bf(d)), 1, N, OC, OC, B_.ptr(sc), nb, None) == 0
    assert rel_l2(host(db), rounded(d).sum(0)) < 1e-6


def _lse_f64(qkv, H):
    """Row log-sum-exp of the causal scaled scores, [B, H, T], in float64."""
    B, T, C3 = qkv.shape
    C = C3 // 3
    hs = C // H
    q = qkv[..., :C].reshape(B, T, H, hs).transpose(0, 2, 1, 3)
    k = qkv[..., C:2 * C].reshape(B, T, H, hs).transpose(0, 2, 1, 3)
    s = q @ k.transpose(0, 1, 3, 2) / np.sqrt(hs)
    s = np.where(np.tril(np.ones((T, T), bool)), s, -np.inf)
    m = s.max(axis=-1, keepdims=True)
    return (m + np.log(np.exp(s - m).sum(axis=-1, keepdims=True)))[..., 0]


@pytest.mark.parametrize("B,T,C,H,ramp", [(1, 300, 768, 12, 0.0), (2, 200, 128, 2, 6.0), (1, 1024, 768, 12, 3.0),
                                          (1, 64, 64, 1, 0.0), (3, 65, 192, 3, 6.0), (2, 384, 128, 2, 6.0),
                                          (1, 513, 64, 1, 3.0), (4, 1024, 128, 2, 0.0)])
def test_bf16_attention_forward_lse(B_, o64, B, T, C, H, ramp):
    """Forward output and log-sum-exp; `ramp` grows the key scale along the
    sequence so the row maxima keep rising across key tiles."""
    L = B_.lib()
    rng = np.random.default_rng(6)
    qkv = rng.normal(size=(B, T, 3 * C))
    qkv[..., C:2 * C] *= (1.0 + ramp * np.arange(T) / T)[None, :, None]
    qr = rounded(qkv)
    y16 = torch.empty(B, T, C, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, H, T, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert L.gpt2_op_attention_forward(B_.ptr(y16), B_.ptr(lse), B_.ptr(bf(qkv)), B, T, C, H, B_.GPT2_MODE_BF16,
                                       B_.ptr(st), None) == 0
    wy, _ = o64.attention_forward(qr, H)
    assert rel_l2(host(y16), wy) < 1e-2
    assert np.abs(host(lse) - _lse_f64(qr, H)).max() < 1e-3 * max(1.0, np.abs(_lse_f64(qr, H)).max())
    assert int(st.item()) == 0


@pytest.mark.parametrize("B,T,C,H", [(2, 37, 64, 4), (1, 300, 768, 12), (2, 129, 192, 3), (1, 1, 64, 4),
                                     (1, 1024, 768, 12), (3, 65, 128, 2), (1, 1, 64, 1)])
def test_bf16_attention(B_, o64, B, T, C, H):
    L = B_.lib()
    rng = np.random.default_rng(5)
    qkv = rng.normal(size=(B, T, 3 * C))
    dy = rng.normal(size=(B, T, C))
    qr, dr = rounded(qkv), rounded(dy)
    q16 = bf(qkv)
    y16 = torch.empty(B, T, C, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, H, T, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert L.gpt2_op_attention_forward(B_.ptr(y16), B_.ptr(lse), B_.ptr(q16), B, T, C, H, B_.GPT2_MODE_BF16,
                                       B_.ptr(st), None) == 0
    wy, P = o64.attention_forward(qr, H)
    assert rel_l2(host(y16), wy) < 1e-2
    dq16 = torch.empty(B, T, 3 * C, dtype=torch.bfloat16, device="cuda")
    nb = L.gpt2_op_attention_backward_scratch_bytes(B, T, H)
    sc = torch.empty(nb, dtype=torch.uint8, device="cuda")
    assert L.gpt2_op_attention_backward(B_.ptr(dq16), B_.ptr(bf(dy)), B_.ptr(q16), B_.ptr(y16), B_.ptr(lse),
                                        B, T, C, H, B_.ptr(sc), nb, B_.GPT2_MODE_BF16, B_.ptr(st), None) == 0
    want = o64.attention_backward(dr, qr, P, H)
    got = host(dq16)
    for i, name in enumerate("qkv"):
        assert rel_l2(got[..., i * C:(i + 1) * C], want[..., i * C:(i + 1) * C]) < 1e-2, name
    assert int(st.item()) == 0
