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


def _check(L, B_, dout, N, OC, ld, rng_call):
    """One no-alloc call against the allocating entry point (the same kernels
    in the same order: bit-equal) and against the column sum."""
    want = _reference(L, B_, dout, N, OC, ld)
    db = torch.full((OC,), float("nan"), device="cuda")
    assert L.gpt2_op_bias_grad_noalloc(B_.ptr(db), B_.ptr(dout), N, OC, ld, None) == 0
    torch.cuda.synchronize()
    got = db.cpu().numpy()
    assert np.array_equal(got, want), rng_call
    cols = dout.view(-1)[: (N - 1) * ld + OC]
    full = torch.nn.functional.pad(cols, (0, N * ld - cols.numel())).view(N, ld)
    assert rel_l2(got, full.double().sum(0)[:OC].cpu().numpy()) < 1e-5


@pytest.mark.parametrize("N,OC,ld", [(16384, 3072, 3072), (300, 65, 128), (1, 7, 7)])
def test_noalloc_bias_grad_matches_allocating_entry_point(N, OC, ld):
    from gpt_decoder_step_train_b300 import binding as B_
    L = B_.lib()
    rng = np.random.default_rng(N + OC)
    # two calls in a row with different inputs: the shared array holds the first
    # call's partials when the second one starts
    for call in range(2):
        dout = torch.from_numpy(rng.normal(size=(N, ld)).astype(np.float32)).cuda()
        _check(L, B_, dout, N, OC, ld, call)


def test_noalloc_bias_grad_at_its_size_limit():
    """Exactly GPT2_BIAS_GRAD_NOALLOC_MAX_PARTIALS partial sums: the last row
    chunk's partials fill the array's last entries."""
    from gpt_decoder_step_train_b300 import binding as B_
    L = B_.lib()
    N, OC = 256 * 1024, 1024
    assert (N + 255) // 256 * OC == B_.BIAS_GRAD_NOALLOC_MAX_PARTIALS
    g = torch.Generator(device="cuda").manual_seed(7)
    for call in range(2):
        dout = torch.randn(N, OC, device="cuda", generator=g)
        _check(L, B_, dout, N, OC, OC, call)
        del dout


def test_noalloc_bias_grad_column_slice_with_unaligned_base():
    """dout one element into a wider matrix (a column slice): 16-byte loads do
    not apply, the result is still the column sum."""
    from gpt_decoder_step_train_b300 import binding as B_
    L = B_.lib()
    N, ld, OC = 1000, 3072, 3071
    base = torch.from_numpy(np.random.default_rng(3).normal(size=(N, ld)).astype(np.float32)).cuda()
    dout = base.view(-1)[1:]
    assert dout.data_ptr() % 16 == 4
    _check(L, B_, dout, N, OC, ld, 0)


def test_noalloc_bias_grad_rejects_sizes_beyond_its_array():
    from gpt_decoder_step_train_b300 import binding as B_
    L = B_.lib()
    N, OC = 256 * 1024, 1025            # 1024 row chunks x 1025 columns > 2^20 partials
    assert (N + 255) // 256 * OC > B_.BIAS_GRAD_NOALLOC_MAX_PARTIALS
    dout = torch.zeros(1, device="cuda")
    db = torch.zeros(OC, device="cuda")
    assert L.gpt2_op_bias_grad_noalloc(B_.ptr(db), B_.ptr(dout), N, OC, OC, None) == B_.GPT2_ENOMEM
