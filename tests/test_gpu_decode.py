"""Autoregressive decoding with the key/value cache, against the oracle: the
logits of position t from gpt2_decode equal the oracle's last-row logits of a
full forward over the prefix 0..t (causality makes the two the same function),
plus greedy and top-k token choice and the call-order rules."""
import numpy as np
import pytest

from gpt_decoder_step_train_b300 import synthetic as syn
from gpu_util import rel_l2

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _oracle_last_logits(o, cfg, params, tok_row, t):
    """Oracle logits of position t from a forward over tok_row[0..t]."""
    om = o.model(cfg.dims(), 1, t + 1, last_only=True)
    seq = np.ascontiguousarray(tok_row[None, :t + 1])
    om.forward(params, seq, seq)                  # targets are not used by the logits
    return om.logits()[0][:cfg.V]


def _decode_all(cfg, params, tok, mode, positions):
    from gpt_decoder_step_train_b300.binding import GPT2
    p = torch.from_numpy(params.copy()).cuda()
    model = GPT2(cfg, p, maxB=tok.shape[0], mode=mode)
    B = tok.shape[0]
    out = torch.empty(B, cfg.V, device="cuda")
    got = {}
    for pos in range(max(positions) + 1):
        col = torch.from_numpy(np.ascontiguousarray(tok[:, pos])).cuda()
        assert model.decode(col, pos, out) == 0
        if pos in positions:
            got[pos] = out.cpu().numpy().copy()
    assert model.status() == 0
    model.close()
    return got


@pytest.mark.parametrize("mode", ["fp32", "bf16"])
def test_decode_logits_equal_prefix_forward_tiny(mode, o64):
    cfg = syn.CONFIGS["tiny"]
    params = syn.init_params(cfg, perturbed=True)
    tok, _ = syn.draw_tokens(cfg)
    T = tok.shape[1]
    got = _decode_all(cfg, params, tok, mode, set(range(T)))
    p64 = params.astype(np.float64)
    for b in range(tok.shape[0]):
        want = np.stack([_oracle_last_logits(o64, cfg, p64, tok[b], t) for t in range(T)])
        have = np.stack([got[t][b] for t in range(T)])
        # fp32 arithmetic in every mode: the strict-fp32 bar
        assert rel_l2(have, want) <= 1e-4, (b, rel_l2(have, want))


def test_decode_logits_equal_prefix_forward_124m(o64):
    cfg = syn.CONFIGS["124M_small"]
    params = syn.init_params(cfg)
    tok, _ = syn.draw_tokens(cfg, B=2, T=12)
    positions = {0, 5, 11}
    got = _decode_all(cfg, params, tok, "bf16", positions)
    p64 = params.astype(np.float64)
    for b in range(2):
        for t in sorted(positions):
            want = _oracle_last_logits(o64, cfg, p64, tok[b], t)
            assert rel_l2(got[t][b], want) <= 1e-4, (b, t)


def test_decode_matches_training_forward_logits():
    """Same model, fp32 mode: decode rows equal the forward's logits position by position."""
    from gpt_decoder_step_train_b300.binding import GPT2
    cfg = syn.CONFIGS["tiny"]
    params = torch.from_numpy(syn.init_params(cfg, perturbed=True)).cuda()
    tok, _ = syn.draw_tokens(cfg)
    B, T = tok.shape
    model = GPT2(cfg, params, mode="fp32")
    model.forward(torch.from_numpy(tok).cuda())                # logits kept
    full = model.logits(B * T).cpu().numpy()[:, :cfg.V].reshape(B, T, cfg.V).copy()
    out = torch.empty(B, cfg.V, device="cuda")
    for pos in range(T):
        assert model.decode(torch.from_numpy(np.ascontiguousarray(tok[:, pos])).cuda(), pos, out) == 0
        assert rel_l2(out.cpu().numpy(), full[:, pos]) <= 1e-5
    model.close()


def test_argmax_picks_first_maximum_and_skips_nan():
    from gpt_decoder_step_train_b300 import binding as B_
    L = B_.lib()
    rng = np.random.default_rng(7)
    N, V, ld = 6, 50257, 50304
    z = rng.normal(size=(N, ld)).astype(np.float32)
    z[1, 100] = z[1, 4000] = 50.0                          # tie: the lower index
    z[2, :] = -np.inf
    z[2, 77] = -1.0
    z[3, :V] = np.nan
    z[4, 9] = np.nan
    z[4, 10] = 40.0
    z[5, V:] = 1e9                                         # padding is not a candidate
    zt = torch.from_numpy(z).cuda()
    out = torch.empty(N, dtype=torch.int32, device="cuda")
    assert L.gpt2_op_argmax(B_.ptr(out), B_.ptr(zt), N, V, ld, None) == 0
    got = out.cpu().numpy()
    want = np.array([np.argmax(z[0, :V]), 100, 77, 0, 10, np.argmax(z[5, :V])])
    assert np.array_equal(got, want)


def test_greedy_generation_is_deterministic_and_feeds_back():
    """Greedy decoding of a few tokens from a prompt: the chosen token is the
    argmax of the logits that decode returned, and two runs agree exactly."""
    from gpt_decoder_step_train_b300 import binding as B_
    from gpt_decoder_step_train_b300.binding import GPT2
    L = B_.lib()
    cfg = syn.CONFIGS["tiny"]
    params = torch.from_numpy(syn.init_params(cfg, perturbed=True)).cuda()
    prompt, _ = syn.draw_tokens(cfg, B=3, T=5)

    def run():
        model = GPT2(cfg, params, maxB=3, mode="tf32")
        out = torch.empty(3, cfg.V, device="cuda")
        nxt = torch.empty(3, dtype=torch.int32, device="cuda")
        seq = [prompt[:, t] for t in range(prompt.shape[1])]
        for pos in range(12):
            col = torch.from_numpy(np.ascontiguousarray(seq[pos])).cuda() if pos < len(seq) else nxt.clone()
            assert model.decode(col, pos, out) == 0
            assert L.gpt2_op_argmax(B_.ptr(nxt), B_.ptr(out), 3, cfg.V, cfg.V, None) == 0
            assert np.array_equal(nxt.cpu().numpy(), np.argmax(out.cpu().numpy(), axis=1))
            if pos + 1 >= len(seq):
                seq.append(nxt.cpu().numpy().copy())
        model.close()
        return np.stack(seq[:12], axis=1)
    a, b = run(), run()
    assert np.array_equal(a, b)
    assert np.array_equal(a[:, :5], prompt)


def test_decode_call_order_and_errors():
    from gpt_decoder_step_train_b300 import binding as B_
    from gpt_decoder_step_train_b300.binding import GPT2
    cfg = syn.CONFIGS["tiny"]
    params = torch.from_numpy(syn.init_params(cfg)).cuda()
    model = GPT2(cfg, params, maxB=4, mode="bf16")
    out = torch.empty(4, cfg.V, device="cuda")
    tok = torch.tensor([1, 2, 3, 4], dtype=torch.int32, device="cuda")
    assert model.decode(tok[:2], 1, out) == B_.GPT2_ESTATE      # must start at 0
    assert model.status() == B_.GPT2_ESTATE
    assert model.decode(tok[:2], 0, out) == 0
    assert model.decode(tok[:3], 1, out) == B_.GPT2_ESTATE      # B changed
    assert model.decode(tok[:2], 2, out) == B_.GPT2_ESTATE      # skipped a position
    assert model.status() == B_.GPT2_ESTATE
    assert model.decode(tok[:2], 1, out) == 0
    assert model.decode(tok[:2], cfg.maxT, out) == B_.GPT2_EINVAL
    assert model.status() == B_.GPT2_EINVAL
    big = torch.zeros(5, dtype=torch.int32, device="cuda")
    assert model.decode(big, 0, out) == B_.GPT2_EINVAL         # more rows than maxB
    model.status()
    bad = torch.tensor([0, cfg.V], dtype=torch.int32, device="cuda")
    assert model.decode(bad, 0, out) == 0                        # reported through the status word
    assert model.status() == B_.GPT2_ETOKEN
    # training still works after decoding
    tt, tg = syn.draw_tokens(cfg)
    loss = model.forward(torch.from_numpy(tt[:4]).cuda(), torch.from_numpy(tg[:4]).cuda())
    assert np.isfinite(loss) and model.backward() == 0
    model.close()


@pytest.mark.parametrize("k", [1, 5, 50, 64])
def test_sample_topk_matches_oracle(k):
    """gpt2_op_sample_topk against the oracle's definition on the same logits and
    draws: the same token, except where a draw sits within 1e-6 of a cumulative
    boundary (fp32 on the GPU, float64 in the oracle), where either neighbour is
    accepted."""
    from gpt_decoder_step_train_b300 import binding as B_
    from oracle import sample_topk
    L = B_.lib()
    rng = np.random.default_rng(13 + k)
    N, V, ld = 12, 50257, 50304
    z = np.zeros((N, ld), dtype=np.float32)
    z[:, :V] = (rng.normal(size=(N, V)) * 2).astype(np.float32)
    z[3, 1000:1000 + 2 * k] = 9.0                          # ties across the cut
    z[4, 5] = np.nan
    z[:, V:] = 1e9                                          # padding is never a candidate
    u = rng.random(N).astype(np.float32)
    zt, ut = torch.from_numpy(z).cuda(), torch.from_numpy(u).cuda()
    out = torch.empty(N, dtype=torch.int32, device="cuda")
    assert L.gpt2_op_sample_topk(B_.ptr(out), B_.ptr(zt), N, V, ld, k, B_.ptr(ut), None) == 0
    got = out.cpu().numpy()
    want, bounds = sample_topk(z[:, :V], k, u.astype(np.float64))
    for n in range(N):
        if got[n] == want[n]:
            continue
        near = [abs(b - u[n]) < 1e-6 for b in bounds[n]]
        assert any(near), (n, got[n], want[n])
    if k == 1:
        assert np.array_equal(got, np.argmax(np.where(np.isnan(z[:, :V]), -np.inf, z[:, :V]), axis=1))
    assert L.gpt2_op_sample_topk(B_.ptr(out), B_.ptr(zt), N, V, ld, 65, B_.ptr(ut), None) == B_.GPT2_EINVAL
    assert L.gpt2_op_sample_topk(B_.ptr(out), B_.ptr(zt), N, V, ld, 0, B_.ptr(ut), None) == B_.GPT2_EINVAL
