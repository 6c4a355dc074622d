"""The stored oracle values used by the full-size GPU parity tests are current:
they were written by tests/expected/make_row_losses.py from the present oracle
source and input generator, cover every row, and are plausible for the
standard initialisation (near ln V: logits start close to zero)."""
import math
import os
import sys

from conftest import ROOT
from gpt_decoder_step_train_b300 import synthetic as syn

sys.path.insert(0, os.path.join(ROOT, "tests", "expected"))
import make_row_losses  # noqa: E402


def test_row_losses_are_current_and_complete():
    sha, vals = make_row_losses.read()
    assert sha == make_row_losses.sources_sha256()
    for name in make_row_losses.CONFIGS:
        cfg = syn.CONFIGS[name]
        for b in range(cfg.B):
            v = vals[(name, b)]
            # N(0, 0.02) weights: logits of std ~0.3, loss ln V plus a small positive term
            assert math.log(cfg.V) < v < math.log(cfg.V) + 0.5, (name, b, v)
