"""ctypes binding of the C ABI in ``include/gpt2.h`` and ``include/gpt2_ops.h``.

Argument marshalling only: every computation runs in ``libgpt2_b300.so``.
Device memory comes from torch tensors (``tensor.data_ptr()``); streams are
torch streams (``stream.cuda_stream``).  Loading fails loudly when the library
has not been built or no CUDA device is present; there is no fallback.
"""
import ctypes as C
import os

from . import synthetic

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgpt2_b300.so")

GPT2_OK, GPT2_EINVAL, GPT2_ENOMEM, GPT2_ECUDA = 0, -1, -2, -3
GPT2_ETOKEN, GPT2_ESTATE, GPT2_ETIMEOUT, GPT2_ENOTSUP = -4, -5, -6, -7
GPT2_MODE_FP32, GPT2_MODE_TF32, GPT2_MODE_BF16 = 0, 1, 2
MODES = {"fp32": GPT2_MODE_FP32, "tf32": GPT2_MODE_TF32, "bf16": GPT2_MODE_BF16}
GPT2_LINEAR_GELU, GPT2_LINEAR_ZERO_PAD = 1, 2
STATUS_BAD_TOKEN, STATUS_BAD_TARGET, STATUS_TIMEOUT = 1, 2, 4
BIAS_GRAD_NOALLOC_MAX_PARTIALS = 1 << 20
TRACE_CLASSES = ("encoder_fwd", "layernorm_fwd", "matmul_fwd", "attention_fwd", "crossentropy",
                 "matmul_bwd_input", "matmul_bwd_weight", "layernorm_bwd", "attention_bwd",
                 "encoder_bwd", "adamw", "other", "bias_grad", "dropout")


class gpt2_gemm_args(C.Structure):
    _fields_ = [("M", C.c_int), ("N", C.c_int), ("K", C.c_int),
                ("A", C.c_void_p), ("lda", C.c_int), ("a_kmajor", C.c_int),
                ("B", C.c_void_p), ("ldb", C.c_int), ("b_kmajor", C.c_int),
                ("bf16", C.c_int),
                ("out", C.c_void_p), ("ldo", C.c_int), ("out_bf16", C.c_int),
                ("out_pre", C.c_void_p), ("bias", C.c_void_p), ("residual", C.c_void_p),
                ("gelu_x", C.c_void_p), ("ldg", C.c_int), ("gelu", C.c_int),
                ("pre_bf16", C.c_int), ("gelu_x_bf16", C.c_int), ("colsum", C.c_void_p)]


class gpt2_config(C.Structure):
    _fields_ = [("V", C.c_int), ("maxT", C.c_int), ("L", C.c_int), ("H", C.c_int), ("C", C.c_int),
                ("maxB", C.c_int), ("mode", C.c_int), ("workspace", C.c_void_p),
                ("workspace_bytes", C.c_size_t), ("stream", C.c_void_p)]


_vp, _i, _f, _sz = C.c_void_p, C.c_int, C.c_float, C.c_size_t
# name -> (restype, argtypes); mirrors the two headers
SIGNATURES = {
    "gpt2_num_params": (_sz, [_vp]),
    "gpt2_workspace_bytes": (_sz, [_vp]),
    "gpt2_create": (_i, [_vp, _vp, _vp]),
    "gpt2_forward": (_f, [_vp, _vp, _vp, _i, _i]),
    "gpt2_eval": (_f, [_vp, _vp, _vp, _i, _i]),
    "gpt2_set_dropout": (_i, [_vp, _f, C.c_ulonglong]),
    "gpt2_decode": (_i, [_vp, _vp, _i, _i, _vp]),
    "gpt2_backward": (_i, [_vp]),
    "gpt2_adamw": (_i, [_vp, _f, _f, _f, _f, _f, _i]),
    "gpt2_destroy": (_i, [_vp]),
    "gpt2_status": (_i, [_vp]),
    "gpt2_wait_probe": (_i, [_vp, _i]),
    "gpt2_strerror": (C.c_char_p, [_i]),
    "gpt2_grads": (_vp, [_vp]),
    "gpt2_adam_m": (_vp, [_vp]),
    "gpt2_adam_v": (_vp, [_vp]),
    "gpt2_logits": (_vp, [_vp, _vp]),
    "gpt2_losses": (_vp, [_vp]),
    "gpt2_activation": (_vp, [_vp, _i, _i]),
    "gpt2_trace_enable": (_i, [_vp, _i]),
    "gpt2_trace_read": (_i, [_vp, _vp, _vp, _i]),
    "gpt2_kernel_launches": (C.c_longlong, []),
    "gpt2_op_encoder_forward": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp]),
    "gpt2_op_encoder_backward_scratch_bytes": (_sz, [_i, _i, _i]),
    "gpt2_op_encoder_backward": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _sz, _vp]),
    "gpt2_op_layernorm_forward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _vp]),
    "gpt2_op_layernorm_forward_bf16": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _vp]),
    "gpt2_op_layernorm_backward_scratch_bytes": (_sz, [_i, _i]),
    "gpt2_op_layernorm_backward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i,
                                        _vp, _sz, _vp, _vp]),
    "gpt2_op_linear_forward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp,
                                    _vp]),
    "gpt2_op_linear_backward_input": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp]),
    "gpt2_op_linear_backward_weight_scratch_bytes": (_sz, [_i, _i, _i, _i]),
    "gpt2_op_linear_backward_weight": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _sz, _i,
                                            _vp, _vp]),
    "gpt2_op_bias_grad_scratch_bytes": (_sz, [_i, _i]),
    "gpt2_op_bias_grad": (_i, [_vp, _vp, _i, _i, _i, _i, _vp, _sz, _vp]),
    "gpt2_op_gemm": (_i, [_vp, _i, _vp, _vp]),
    "gpt2_op_to_bf16": (_i, [_vp, _vp, _sz, _vp]),
    "gpt2_op_bias_grad_noalloc": (_i, [_vp, _vp, _i, _i, _i, _vp]),
    "gpt2_op_attention_forward": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp]),
    "gpt2_op_attention_backward_scratch_bytes": (_sz, [_i, _i, _i]),
    "gpt2_op_attention_backward": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _sz, _i,
                                        _vp, _vp]),
    "gpt2_op_attention_forward_dropout": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _f, _vp, _vp]),
    "gpt2_op_attention_backward_dropout": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _sz, _i,
                                                _vp, _f, _vp, _vp]),
    "gpt2_op_dropout_mask_words": (_sz, [C.c_longlong, _i]),
    "gpt2_op_dropout_mask": (_i, [_vp, C.c_longlong, _i, _i, C.c_ulonglong, C.c_uint, C.c_uint, _f, _vp]),
    "gpt2_op_dropout_residual": (_i, [_vp, _vp, _vp, _i, _i, _f, _vp]),
    "gpt2_op_dropout_backward": (_i, [_vp, _i, _vp, _vp, _i, _i, _f, _vp]),
    "gpt2_op_layernorm_backward_dropout": (_i, [_vp, _vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i,
                                                _vp, _f, _vp, _sz, _vp, _vp]),
    "gpt2_op_crossentropy": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _f, _vp, _vp]),
    "gpt2_op_crossentropy_bf16": (_i, [_vp, _vp, _vp, _i, _i, _i, _f, _vp, _vp]),
    "gpt2_op_argmax": (_i, [_vp, _vp, _i, _i, _i, _vp]),
    "gpt2_op_sample_topk": (_i, [_vp, _vp, _i, _i, _i, _i, _vp, _vp]),
    "gpt2_op_sum": (_i, [_vp, _vp, _i, _f, _vp]),
    "gpt2_op_adamw": (_i, [_vp, _vp, _vp, _vp, _sz, _f, _f, _f, _f, _f, _f, _f, _vp]),
}

_lib = None


def lib():
    """Load the library (once) and declare every exported function."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: run `python -m gpt_decoder_step_train_b300.build`")
    L = C.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def strerror(code):
    return lib().gpt2_strerror(code).decode()


def check(code, what=""):
    if code != GPT2_OK:
        raise RuntimeError(f"{what} failed: {code} ({strerror(code)})")


def ptr(t):
    """Device (or host) address of a torch tensor, or None."""
    return None if t is None else C.c_void_p(t.data_ptr())


def stream_handle(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def make_config(cfg, maxB=None, mode="tf32", workspace=None, workspace_bytes=0, stream=None):
    c = gpt2_config()
    c.V, c.maxT, c.L, c.H, c.C = cfg.V, cfg.maxT, cfg.L, cfg.H, cfg.C
    c.maxB = cfg.B if maxB is None else maxB
    c.mode = MODES[mode] if isinstance(mode, str) else int(mode)
    c.workspace = workspace
    c.workspace_bytes = workspace_bytes
    c.stream = stream
    return c


class GPT2:
    """One model over a caller-owned flat fp32 parameter tensor on the GPU.

    The workspace is a torch uint8 tensor, so every buffer the library hands
    back (gradients, moments, logits, activations) is exposed as a view of it.
    """

    def __init__(self, cfg, params, maxB=None, mode="tf32", stream=None):
        import torch
        L = lib()
        self.cfg = cfg
        self.mode = mode
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        self.params = params
        assert params.is_cuda and params.dtype == torch.float32 and params.is_contiguous()
        probe = make_config(cfg, maxB, mode)
        self.nparams = L.gpt2_num_params(C.byref(probe))
        if self.nparams == 0:
            raise ValueError("invalid configuration")
        assert params.numel() == self.nparams == synthetic.num_params(cfg)
        nbytes = L.gpt2_workspace_bytes(C.byref(probe))
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=params.device)
        self.c = make_config(cfg, maxB, mode, C.c_void_p(self.workspace.data_ptr()), nbytes,
                             C.c_void_p(self.stream.cuda_stream))
        h = C.c_void_p()
        check(L.gpt2_create(C.byref(self.c), ptr(params), C.byref(h)), "gpt2_create")
        self.h = h

    def close(self):
        if getattr(self, "h", None):
            lib().gpt2_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- the four calls of the step --------------------------------------
    def forward(self, tokens, targets=None):
        B, T = tokens.shape
        return lib().gpt2_forward(self.h, ptr(tokens), ptr(targets), B, T)

    def eval(self, tokens, targets):
        """Mean loss only (no gradient of the logits is left for a backward)."""
        B, T = tokens.shape
        return lib().gpt2_eval(self.h, ptr(tokens), ptr(targets), B, T)

    def decode(self, tokens, pos, logits):
        """Advance len(tokens) sequences by one position; logits [B, V] (device) receives the new row."""
        return lib().gpt2_decode(self.h, ptr(tokens), int(tokens.shape[0]), pos, ptr(logits))

    def set_dropout(self, p, seed=0):
        """Dropout with probability p for the following training forwards (0: off)."""
        return lib().gpt2_set_dropout(self.h, float(p), int(seed))

    def backward(self):
        return lib().gpt2_backward(self.h)

    def adamw(self, lr, b1, b2, eps, wd, t):
        return lib().gpt2_adamw(self.h, lr, b1, b2, eps, wd, t)

    def status(self):
        return lib().gpt2_status(self.h)

    def trace(self, on=True):
        check(lib().gpt2_trace_enable(self.h, int(on)), "gpt2_trace_enable")

    def trace_read(self):
        """{class name: (milliseconds, kernel launches)} since the last read."""
        n = len(TRACE_CLASSES)
        ms = (C.c_double * n)()
        nl = (C.c_longlong * n)()
        check(lib().gpt2_trace_read(self.h, C.cast(ms, C.c_void_p), C.cast(nl, C.c_void_p), n),
              "gpt2_trace_read")
        return {name: (ms[i], nl[i]) for i, name in enumerate(TRACE_CLASSES)}

    # -- views into the workspace ----------------------------------------
    def _view(self, addr, n, shape=None, bf16=False):
        import torch
        es = 2 if bf16 else 4
        off = addr - self.workspace.data_ptr()
        assert 0 <= off and off + es * n <= self.workspace.numel()
        t = self.workspace[off:off + es * n].view(torch.bfloat16 if bf16 else torch.float32)
        return t.view(*shape) if shape else t

    def grads(self):
        return self._view(lib().gpt2_grads(self.h), self.nparams)

    def adam_m(self):
        return self._view(lib().gpt2_adam_m(self.h), self.nparams)

    def adam_v(self):
        return self._view(lib().gpt2_adam_v(self.h), self.nparams)

    def logits(self, rows):
        ld = C.c_int()
        a = lib().gpt2_logits(self.h, C.byref(ld))
        return self._view(a, rows * ld.value, (rows, ld.value))

    def losses(self, rows):
        return self._view(lib().gpt2_losses(self.h), rows)

    # activations held as bf16 in bf16 mode (the tensor-core operands)
    BF16_ACTIVATIONS = (1, 2, 3, 5, 6, 7, 9)

    def activation(self, which, layer, rows):
        """Activation `which` of block `layer` as a [rows, width] view (bf16 or fp32)."""
        widths = {0: 1, 1: 1, 2: 3, 3: 1, 4: 1, 5: 1, 6: 4, 7: 4, 8: 1, 9: 1}
        w = widths[which] * self.cfg.C
        a = lib().gpt2_activation(self.h, which, layer)
        return self._view(a, rows * w, (rows, w), bf16=self.mode == "bf16" and which in self.BF16_ACTIVATIONS)
