"""The allocation-free bias gradient gives the same result as the allocating
entry point.

Some callers cannot call cudaMalloc (a host application that owns the device
memory budget and hands a plugin only its input and output buffers, or a loop
that plans all memory at start-up); gpt2_op_bias_grad_noalloc serves them with
a fixed array inside the library.  This file is collected last, and passes both
on its own in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest

from gpu_util import rel_l2

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _reference(L, B_, dout, N, OC, ld):
    db = torch.empty(OC, device="cuda")
    nbytes = L.gpt2_op_bias_grad_scratch_bytes(N, OC)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    assert L.gpt2_op_bias_grad(B_.ptr(db), B_.ptr(dout), 0, N, OC, ld, B_.ptr(scratch), nbytes,
                               None) == 0
    torch.cuda.synchronize()
    return db.cpu().numpy()


@pytest.mark.parametrize("N,OC,ld", [(16384, 3072, 3072), (300, 65, 128), (1, 7, 7)])
def test_noalloc_bias_grad_matches_allocating_entry_point(N, OC, ld):
    from gpt_decoder_step_train_b300 import binding as B_
    L = B_.lib()
    rng = np.random.default_rng(N + OC)
    # two calls in a row with different inputs: the shared array holds the first
    # call's partials when the second one starts
    for call in range(2):
        dout = torch.from_numpy(rng.normal(size=(N, ld)).astype(np.float32)).cuda()
        want = _reference(L, B_, dout, N, OC, ld)
        db = torch.full((OC,), float("nan"), device="cuda")
        assert L.gpt2_op_bias_grad_noalloc(B_.ptr(db), B_.ptr(dout), N, OC, ld, None) == 0
        torch.cuda.synchronize()
        got = db.cpu().numpy()
        assert rel_l2(got, want) < 1e-6, call
        # the oracle-free property: the bias gradient is the column sum
        assert rel_l2(got, dout.double().sum(0)[:OC].cpu().numpy()) < 1e-5


def test_noalloc_bias_grad_rejects_sizes_beyond_its_array():
    from gpt_decoder_step_train_b300 import binding as B_
    L = B_.lib()
    N, OC = 256 * 1024, 1025            # 1024 row chunks x 1025 columns > 2^20 partials
    assert (N + 255) // 256 * OC > B_.BIAS_GRAD_NOALLOC_MAX_PARTIALS
    dout = torch.zeros(1, device="cuda")
    db = torch.zeros(OC, device="cuda")
    assert L.gpt2_op_bias_grad_noalloc(B_.ptr(db), B_.ptr(dout), N, OC, OC, None) == B_.GPT2_ENOMEM
