"""The C-ABI library loads, exports every symbol the headers declare, and its
host-only calls work without a GPU."""
import ctypes
import os
import re

import pytest

from conftest import ROOT
from gpt_decoder_step_train_b300 import synthetic as syn

HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


def declared_functions():
    names = set()
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"\b(gpt2_[a-z0-9_]+)\s*\(", src):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def L():
    from gpt_decoder_step_train_b300 import binding
    return binding.lib()


def test_headers_declare_the_four_step_calls():
    names = declared_functions()
    for n in ("gpt2_create", "gpt2_forward", "gpt2_backward", "gpt2_adamw"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in sorted(declared_functions()) if not hasattr(L, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    from gpt_decoder_step_train_b300 import binding
    assert declared_functions() == set(binding.SIGNATURES)


def _dynamic_symbols(path, which):
    import subprocess
    r = subprocess.run(["nm", "-D", which, path], capture_output=True, text=True, check=True)
    return [line.split()[-1] for line in r.stdout.splitlines() if line.strip()]


def test_library_links_no_oracle_code():
    """Neither the symbols the library defines nor those it needs from other
    libraries name the oracle, and it links no oracle library (read from the
    dynamic symbol table and the DT_NEEDED entries, not from the file's bytes)."""
    import subprocess
    from gpt_decoder_step_train_b300 import binding
    defined = _dynamic_symbols(binding.LIB_PATH, "--defined-only")
    undefined = _dynamic_symbols(binding.LIB_PATH, "--undefined-only")
    assert "gpt2_create" in defined and undefined
    assert not [s for s in defined + undefined if "oracle" in s.lower()]
    dyn = subprocess.run(["readelf", "-d", binding.LIB_PATH], capture_output=True, text=True, check=True).stdout
    needed = [line for line in dyn.splitlines() if "(NEEDED)" in line]
    assert needed and not [line for line in needed if "oracle" in line.lower()]


@pytest.mark.parametrize("name", list(syn.CONFIGS))
def test_num_params_matches_layout(L, name):
    from gpt_decoder_step_train_b300 import binding
    cfg = syn.CONFIGS[name]
    c = binding.make_config(cfg)
    assert L.gpt2_num_params(ctypes.byref(c)) == syn.num_params(cfg)
    ws = L.gpt2_workspace_bytes(ctypes.byref(c))
    # at least gradients and both moments, well inside one B300's memory
    assert 3 * 4 * syn.num_params(cfg) < ws < 200 * 2**30


def test_invalid_configs_are_rejected(L):
    from gpt_decoder_step_train_b300 import binding
    cfg = syn.CONFIGS["tiny"]
    for bad in (dict(H=3), dict(C=62, H=2), dict(V=0), dict(L=0), dict(maxT=0)):
        c = binding.make_config(cfg.with_(**bad))
        assert L.gpt2_num_params(ctypes.byref(c)) == 0
        assert L.gpt2_workspace_bytes(ctypes.byref(c)) == 0
    c = binding.make_config(cfg, mode=7)
    assert L.gpt2_num_params(ctypes.byref(c)) == 0
    h = ctypes.c_void_p()
    assert L.gpt2_create(ctypes.byref(binding.make_config(cfg)), None, ctypes.byref(h)) == -1
    assert h.value is None


def test_strerror_covers_codes(L):
    from gpt_decoder_step_train_b300 import binding
    for code in range(0, -8, -1):
        assert binding.strerror(code) != "unknown status"


def test_scratch_queries_are_host_only(L):
    assert L.gpt2_op_layernorm_backward_scratch_bytes(16384, 768) > 0
    assert L.gpt2_op_encoder_backward_scratch_bytes(16384, 50257, 768) > 0
    assert L.gpt2_op_attention_backward_scratch_bytes(16, 1024, 12) >= 16 * 12 * 1024 * 4
    assert L.gpt2_op_linear_backward_weight_scratch_bytes(16384, 768, 3072, 1) > 0


def test_dropout_host_logic(L):
    """Mask sizes and argument checks of the dropout calls, which return before
    any device work (no GPU needed)."""
    from gpt_decoder_step_train_b300 import binding as B_
    words = L.gpt2_op_dropout_mask_words
    assert words(37, 100) == 37 * 4            # ceil(100 / 32) words per row
    assert words(16 * 12 * 1024, 1024) == 16 * 12 * 1024 * 32
    assert words(5, 32) == 5 and words(5, 33) == 10 and words(0, 7) == 0
    assert words(-1, 7) == 0 and words(3, 0) == 0
    fake = ctypes.c_void_p(16)                 # never dereferenced: every call below is rejected
    mask = L.gpt2_op_dropout_mask
    assert mask(None, 4, 8, 0, 1, 0, 0, 0.1, None) == B_.GPT2_EINVAL
    assert mask(fake, 4, 8, 0, 1, 0, 0, 1.0, None) == B_.GPT2_EINVAL          # p must be below 1
    assert mask(fake, 4, 8, 0, 1, 0, 0, -0.01, None) == B_.GPT2_EINVAL
    assert mask(fake, 10, 7, 7, 1, 0, 0, 0.1, None) == B_.GPT2_EINVAL         # rows not a multiple of T
    assert mask(fake, 14, 8, 7, 1, 0, 0, 0.1, None) == B_.GPT2_EINVAL         # cols != T
    res = L.gpt2_op_dropout_residual
    assert res(fake, None, fake, 4, 6, 0.1, None) == B_.GPT2_EINVAL          # C % 4
    assert res(ctypes.c_void_p(20), None, fake, 4, 8, 0.1, None) == B_.GPT2_EINVAL   # alignment
    bwd = L.gpt2_op_dropout_backward
    assert bwd(fake, 0, fake, fake, 4, 8, 1.5, None) == B_.GPT2_EINVAL
    assert bwd(ctypes.c_void_p(24), 0, fake, fake, 4, 8, 0.1, None) == B_.GPT2_EINVAL  # fp32 dst 16 B
    assert L.gpt2_set_dropout(None, 0.1, 0) == B_.GPT2_EINVAL
    assert L.gpt2_op_attention_forward_dropout(fake, fake, fake, 1, 8, 64, 1, B_.GPT2_MODE_BF16, None, 0.1,
                                               None, None) == B_.GPT2_EINVAL  # bits required


def test_missing_library_fails_loudly():
    """Without the built CUDA library the binding raises; there is no fallback."""
    import subprocess
    import sys
    code = ("import gpt_decoder_step_train_b300.binding as b\n"
            "b.LIB_PATH = '/nonexistent/libgpt2_b300.so'\n"
            "b._lib = None\n"
            "try:\n    b.lib()\nexcept RuntimeError as e:\n    print('raised', 'missing' in str(e))\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True, timeout=120)
    assert r.stdout.strip() == "raised True", (r.stdout, r.stderr[-1000:])
