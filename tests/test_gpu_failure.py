"""Failure detection on the GPU without a fault: a bounded device wait that
runs out returns an error status through gpt2_status, and the model keeps
working.  The wait is the one every tensor-core and bulk-copy kernel uses; here
it waits on barriers that nothing completes (gpt2_wait_probe), so it must give
up by its limit."""
import time

import numpy as np
import pytest

from gpt_decoder_step_train_b300 import synthetic as syn

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def test_bounded_wait_runs_out_and_the_model_recovers():
    from gpt_decoder_step_train_b300 import binding as B_
    from gpt_decoder_step_train_b300.binding import GPT2
    cfg = syn.CONFIGS["tiny"]
    params = torch.from_numpy(syn.init_params(cfg)).cuda()
    tok, tgt = syn.draw_tokens(cfg)
    t_tok, t_tgt = torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda()
    model = GPT2(cfg, params, mode="bf16")
    ref = model.forward(t_tok, t_tgt)
    assert np.isfinite(ref) and model.status() == 0
    L = B_.lib()
    assert L.gpt2_wait_probe(model.h, 0) == B_.GPT2_EINVAL
    assert L.gpt2_wait_probe(model.h, 2_000_000) == B_.GPT2_EINVAL
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert L.gpt2_wait_probe(model.h, 1000) == 0          # 1 ms limit
    assert model.status() == B_.GPT2_ETIMEOUT              # synchronises, reads and clears
    elapsed = time.perf_counter() - t0
    # the second wait (one-second limit) left on the first one's abort flag
    assert elapsed < 0.5, elapsed
    assert model.status() == 0                             # cleared
    # the context and the model still work: the same step gives the same loss
    assert model.forward(t_tok, t_tgt) == ref
    assert model.backward() == 0 and model.status() == 0
    model.close()
