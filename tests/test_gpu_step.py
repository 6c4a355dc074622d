"""Whole-step parity: forward + backward + AdamW through the C ABI against the
oracle on the same seeded inputs, per tensor; plus determinism, resume and
error reporting."""
import functools

import numpy as np
import pytest

from gpt_decoder_step_train_b300 import synthetic as syn
from gpu_util import TOL, gpu_steps, oracle_steps, per_tensor, rel_l2

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

# shape coverage: head size 8, odd vocabulary, T not a power of two; lr of the tiny config
RAGGED = syn.Config("ragged-V97-L3-H6-C48-B3T19", V=97, maxT=24, L=3, H=6, C=48, B=3, T=19,
                    lr=1e-4, wd=0.1)
CASES = {
    "tiny": (syn.CONFIGS["tiny"], 3),
    "ragged": (RAGGED, 3),
    "124M_small": (syn.CONFIGS["124M_small"], 1),
}


@functools.lru_cache(maxsize=None)
def oracle_result(name, perturbed):
    from oracle import Oracle
    cfg, steps = CASES[name]
    params = syn.init_params(cfg, perturbed=perturbed)
    tok, tgt = syn.draw_tokens(cfg)
    return oracle_steps(Oracle("f64"), cfg, params.astype(np.float64), tok, tgt, steps)


def _worst(errs, k=4):
    return dict(sorted(errs.items(), key=lambda kv: -kv[1])[:k])


@pytest.mark.parametrize("init", ["standard", "perturbed"])
@pytest.mark.parametrize("mode", ["fp32", "tf32", "bf16"])
@pytest.mark.parametrize("name", list(CASES))
def test_step_matches_oracle(name, mode, init):
    """Loss at every step, every gradient tensor at step 1, and the parameters
    after the last AdamW step, per tensor, within the mode's bar."""
    cfg, steps = CASES[name]
    if name == "124M_small" and init == "perturbed" and mode == "fp32":
        pytest.skip("one perturbed 124M case (tf32) keeps the CPU time of the suite bounded")
    if mode == "bf16" and (cfg.C // cfg.H) not in (16, 32, 64):
        pytest.skip("the bf16 attention kernels take head sizes 16, 32 and 64")
    perturbed = init == "perturbed"
    params = syn.init_params(cfg, perturbed=perturbed)
    tok, tgt = syn.draw_tokens(cfg)
    g_losses, g_grads, g_params = gpu_steps(cfg, params, tok, tgt, mode, steps)
    o_losses, o_grads, o_params = oracle_result(name, perturbed)
    tol = TOL[mode]
    for a, b in zip(g_losses, o_losses):
        assert abs(a - b) <= tol["loss"], (g_losses, o_losses)
    gt, ot = per_tensor(cfg, g_grads), per_tensor(cfg, o_grads)
    errs = {k: rel_l2(gt[k], ot[k]) for k in gt}
    assert max(errs.values()) <= tol["rel"], _worst(errs)
    assert rel_l2(g_params, o_params) <= tol["rel"]
    pt, po = per_tensor(cfg, g_params), per_tensor(cfg, o_params)
    # The key bias (columns C..2C of qkvb) has an identically zero gradient: it adds
    # q_i . b_k to every score of row i, and the softmax ignores a row constant.  Adam
    # divides that rounding noise by its own magnitude, so the key-bias update is
    # O(lr) noise in any finite precision (the oracle's own fp32 build misses 1e-4
    # there).  Those entries are checked apart: gradient at noise level, bounded step.
    C, L = cfg.C, cfg.L
    qb_g, qb_o = pt["qkvb"].reshape(L, 3 * C), po["qkvb"].reshape(L, 3 * C)
    pt["qkvb"] = np.concatenate([qb_g[:, :C], qb_g[:, 2 * C:]], 1)
    po["qkvb"] = np.concatenate([qb_o[:, :C], qb_o[:, 2 * C:]], 1)
    # A tensor that starts at exactly zero holds, after the first AdamW steps,
    # lr * m/(sqrt(v)+eps) ~ -lr * sign(g): a discontinuous function of g, so wherever
    # |g| is below the arithmetic's gradient error its sign is noise.  Those tensors
    # meet the bar from the perturbed init (non-zero start); from the standard init
    # they are left to the whole-vector check above.
    skip = set(syn.ZERO_INIT) if not perturbed else set()
    perrs = {k: rel_l2(pt[k], po[k]) for k in pt if k not in skip}
    assert max(perrs.values()) <= tol["rel"], _worst(perrs)
    kb_grad = gt["qkvb"].reshape(L, 3 * C)[:, C:2 * C]
    q_grad_rms = np.sqrt(np.mean(ot["qkvb"].reshape(L, 3 * C)[:, :C] ** 2))
    # at the arithmetic's noise level: 1e-3 of a typical bias gradient in fp32, 1e-1 in tf32
    assert np.abs(kb_grad).max() <= 10 * tol["rel"] * q_grad_rms
    kb0 = syn.init_params(cfg, perturbed=perturbed)[syn.tensor_offsets(cfg)["qkvb"][0]:][:L * 3 * C]
    kb0 = kb0.reshape(L, 3 * C)[:, C:2 * C]
    assert np.abs(qb_g[:, C:2 * C] - kb0).max() <= cfg.lr * steps * 1.0001 + cfg.wd * cfg.lr * steps


@pytest.mark.parametrize("mode", ["fp32", "tf32", "bf16"])
def test_logits_match_oracle(mode, o64):
    from gpt_decoder_step_train_b300.binding import GPT2
    # bf16 attention takes head sizes 16, 32 and 64
    cfg = RAGGED.with_(H=3) if mode == "bf16" else RAGGED
    params = syn.init_params(cfg)
    tok, tgt = syn.draw_tokens(cfg)
    m = o64.model(cfg.dims(), cfg.B, cfg.T)
    m.forward(params.astype(np.float64), tok, tgt)
    p = torch.from_numpy(params).cuda()
    model = GPT2(cfg, p, mode=mode)
    loss = model.forward(torch.from_numpy(tok).cuda())        # no targets: logits are kept
    assert np.isnan(loss) and model.status() == 0
    z = model.logits(cfg.B * cfg.T).cpu().numpy()
    assert rel_l2(z[:, :cfg.V], m.logits()) <= TOL[mode]["rel"]
    assert np.all(z[:, cfg.V:] == 0)
    # intermediate activations of the first block
    for which, name in [(1, "ln1"), (2, "qkv"), (3, "atty"), (4, "res2"), (6, "h"), (7, "g")]:
        a = model.activation(which, 0, cfg.B * cfg.T).float().cpu().numpy()
        assert rel_l2(a, m.act(name, 0)) <= TOL[mode]["rel"], name
    model.close()


@pytest.mark.parametrize("mode", ["fp32", "tf32", "bf16"])
def test_step_is_deterministic(mode):
    cfg = syn.CONFIGS["tiny"]
    params = syn.init_params(cfg)
    tok, tgt = syn.draw_tokens(cfg)
    a = gpu_steps(cfg, params, tok, tgt, mode, 2)
    b = gpu_steps(cfg, params, tok, tgt, mode, 2)
    assert a[0] == b[0]
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])


def test_resume_from_saved_state_equals_straight_run():
    """Save (params, m, v) after 2 steps, restore into a fresh model, run 2 more:
    identical to 4 straight steps."""
    from gpt_decoder_step_train_b300.binding import GPT2
    cfg = RAGGED
    params = syn.init_params(cfg)
    tok, tgt = syn.draw_tokens(cfg)
    t_tok, t_tgt = torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda()

    def run(model, t0, t1):
        for t in range(t0, t1):
            model.forward(t_tok, t_tgt)
            assert model.backward() == 0
            assert model.adamw(cfg.lr, cfg.b1, cfg.b2, cfg.eps, cfg.wd, t) == 0

    p1 = torch.from_numpy(params.copy()).cuda()
    m1 = GPT2(cfg, p1, mode="tf32")
    run(m1, 1, 5)
    straight = p1.cpu().numpy()

    p2 = torch.from_numpy(params.copy()).cuda()
    m2 = GPT2(cfg, p2, mode="tf32")
    run(m2, 1, 3)
    saved = (p2.clone(), m2.adam_m().clone(), m2.adam_v().clone())
    m2.close()
    p3 = saved[0].clone()
    m3 = GPT2(cfg, p3, mode="tf32")
    m3.adam_m().copy_(saved[1])
    m3.adam_v().copy_(saved[2])
    run(m3, 3, 5)
    assert np.array_equal(p3.cpu().numpy(), straight)


def test_errors_are_reported_not_trapped():
    from gpt_decoder_step_train_b300 import binding as B_
    from gpt_decoder_step_train_b300.binding import GPT2
    cfg = syn.CONFIGS["tiny"]
    params = torch.from_numpy(syn.init_params(cfg)).cuda()
    model = GPT2(cfg, params, mode="fp32")
    tok, tgt = syn.draw_tokens(cfg)
    # backward before any forward
    assert model.backward() == B_.GPT2_ESTATE
    assert model.status() == B_.GPT2_ESTATE
    # adamw before a backward
    assert model.adamw(1e-3, 0.9, 0.999, 1e-8, 0.0, 1) == B_.GPT2_ESTATE
    assert model.status() == B_.GPT2_ESTATE
    # token id out of range
    bad = tok.copy()
    bad[1, 3] = cfg.V
    assert np.isnan(model.forward(torch.from_numpy(bad).cuda(), torch.from_numpy(tgt).cuda()))
    assert model.status() == B_.GPT2_ETOKEN
    # target id out of range
    badt = tgt.copy()
    badt[0, 0] = -1
    assert np.isnan(model.forward(torch.from_numpy(tok).cuda(), torch.from_numpy(badt).cuda()))
    assert model.status() == B_.GPT2_ETOKEN
    # T beyond the context length
    long_tok = np.zeros((1, cfg.maxT + 1), dtype=np.int32)
    assert np.isnan(model.forward(torch.from_numpy(long_tok).cuda()))
    assert model.status() == B_.GPT2_EINVAL
    # the model still works afterwards
    loss = model.forward(torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda())
    assert np.isfinite(loss) and model.status() == 0
    assert model.backward() == 0
    model.close()


def test_host_token_buffers_give_same_loss():
    from gpt_decoder_step_train_b300.binding import GPT2
    cfg = RAGGED
    params = torch.from_numpy(syn.init_params(cfg)).cuda()
    tok, tgt = syn.draw_tokens(cfg)
    model = GPT2(cfg, params, mode="tf32")
    a = model.forward(torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda())
    b = model.forward(torch.from_numpy(tok).pin_memory(), torch.from_numpy(tgt).pin_memory())
    c = model.forward(torch.from_numpy(tok), torch.from_numpy(tgt))   # pageable
    assert a == b == c
    model.close()


@pytest.mark.parametrize("mode", ["fp32", "tf32", "bf16"])
def test_eval_gives_the_forward_loss_and_no_gradient(mode):
    """gpt2_eval: the same mean loss as the training forward (bit for bit: the
    cross-entropy only skips its gradient pass), no backward after it, and in the
    fp32 modes the logits are left as a forward without targets leaves them."""
    from gpt_decoder_step_train_b300 import binding as B_
    from gpt_decoder_step_train_b300.binding import GPT2
    cfg = syn.CONFIGS["tiny"]
    params = torch.from_numpy(syn.init_params(cfg)).cuda()
    tok, tgt = syn.draw_tokens(cfg)
    t_tok, t_tgt = torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda()
    model = GPT2(cfg, params, mode=mode)
    train = model.forward(t_tok, t_tgt)
    ev = model.eval(t_tok, t_tgt)
    assert ev == train and np.isfinite(ev)
    assert model.backward() == B_.GPT2_ESTATE
    assert model.status() == B_.GPT2_ESTATE
    if mode != "bf16":
        z_eval = model.logits(cfg.B * cfg.T).cpu().numpy().copy()
        model.forward(t_tok)                                   # no targets: logits kept
        assert np.array_equal(model.logits(cfg.B * cfg.T).cpu().numpy(), z_eval)
    # targets are required
    assert np.isnan(model.eval(t_tok, None))
    assert model.status() == B_.GPT2_EINVAL
    # a training forward after an eval still trains
    assert model.forward(t_tok, t_tgt) == train
    assert model.backward() == 0
    model.close()


@pytest.mark.parametrize("mode", ["fp32", "tf32", "bf16"])
@pytest.mark.parametrize("name", ["tiny", "124M_small"])
def test_eval_matches_oracle(name, mode):
    """gpt2_eval (forward-only evaluation, no gradient) against the oracle's
    forward on the same inputs: the mean loss within the mode's loss bar, and
    the per-position losses within its relative bar."""
    from gpt_decoder_step_train_b300.binding import GPT2
    cfg, _ = CASES[name]
    o_losses, _, _ = oracle_result(name, False)
    params = syn.init_params(cfg)
    tok, tgt = syn.draw_tokens(cfg)
    p = torch.from_numpy(params.copy()).cuda()
    model = GPT2(cfg, p, mode=mode)
    ev = model.eval(torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda())
    assert model.status() == 0 and np.isfinite(ev)
    assert abs(ev - o_losses[0]) <= TOL[mode]["loss"], (ev, o_losses[0])
    g_pos = model.losses(cfg.B * cfg.T).cpu().numpy()
    from oracle import Oracle
    om = Oracle("f64").model(cfg.dims(), cfg.B, cfg.T)
    om.forward(params.astype(np.float64), tok, tgt)
    assert rel_l2(g_pos, om.losses()) <= TOL[mode]["rel"]
    # evaluation leaves the parameters as they were
    assert np.array_equal(p.cpu().numpy(), params)
    model.close()
