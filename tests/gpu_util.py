"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and compare with the oracle, tensor by tensor."""
import numpy as np

from gpt_decoder_step_train_b300 import synthetic as syn

# parity bars: strict fp32 mode and tensor-core (tf32) mode
TOL = {
    "fp32": {"loss": 1e-4, "rel": 1e-4},
    "tf32": {"loss": 2e-3, "rel": 1e-2},
    "bf16": {"loss": 2e-3, "rel": 1e-2},
}


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def per_tensor(cfg, flat):
    out = {}
    for name, (off, n) in syn.tensor_offsets(cfg).items():
        out[name] = flat[off:off + n]
    return out


def gpu_steps(cfg, params32, tok, tgt, mode, steps=1, maxB=None, lr=None, wd=None):
    """Run `steps` fwd+bwd+AdamW steps through the C ABI on one fixed batch.
    Returns (losses, grads of step 1, logits-free params after the last step)."""
    import torch
    from gpt_decoder_step_train_b300.binding import GPT2
    dev = torch.device("cuda")
    p = torch.from_numpy(params32.copy()).to(dev)
    model = GPT2(cfg, p, maxB=maxB or tok.shape[0], mode=mode)
    t_tok = torch.from_numpy(tok).to(dev)
    t_tgt = torch.from_numpy(tgt).to(dev)
    lr = cfg.lr if lr is None else lr
    wd = cfg.wd if wd is None else wd
    losses, grads1 = [], None
    for t in range(1, steps + 1):
        loss = model.forward(t_tok, t_tgt)
        assert model.status() == 0
        losses.append(loss)
        assert model.backward() == 0
        if t == 1:
            grads1 = model.grads().cpu().numpy().copy()
        assert model.adamw(lr, cfg.b1, cfg.b2, cfg.eps, wd, t) == 0
    assert model.status() == 0
    out = p.cpu().numpy().copy()
    model.close()
    return losses, grads1, out


def oracle_steps(o, cfg, params, tok, tgt, steps=1, lr=None, wd=None):
    lr = cfg.lr if lr is None else lr
    wd = cfg.wd if wd is None else wd
    m = o.model(cfg.dims(), tok.shape[0], tok.shape[1])
    p = params.astype(o.dtype).copy()
    am, av = np.zeros_like(p), np.zeros_like(p)
    losses, grads1 = [], None
    for t in range(1, steps + 1):
        losses.append(m.forward(p, tok, tgt))
        g = m.backward(p)
        if t == 1:
            grads1 = g.copy()
        m.adamw(p, g, am, av, lr, cfg.b1, cfg.b2, cfg.eps, wd, t)
    return losses, grads1, p
