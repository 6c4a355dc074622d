"""Write fullsize_row_mean_loss.txt: the oracle's mean cross-entropy of every
row (sequence) of the full-size workloads, for the GPU parity tests.

Calls only the oracle (double-precision build) on the seeded inputs of
``gpt_decoder_step_train_b300.synthetic``; nothing here runs the CUDA path.
Each row is an independent forward of B = 1 (a row's loss depends on that row
only), so the values equal the per-row means of one forward over the batch.
The file records the sha256 of the oracle source and of the input generator,
and the tests refuse a file whose hashes no longer match.

Usage: python tests/expected/make_row_losses.py [config ...]   (default: all
three full-size configurations; about an hour on 8 cores)
"""
import hashlib
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

from gpt_decoder_step_train_b300 import synthetic as syn  # noqa: E402
from oracle import Oracle  # noqa: E402

OUT = os.path.join(HERE, "fullsize_row_mean_loss.txt")
CONFIGS = ("124M", "350M", "1.5B")
HASHED = ("oracle/gpt2_oracle.c", "gpt_decoder_step_train_b300/synthetic.py")


def sources_sha256():
    h = hashlib.sha256()
    for f in HASHED:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()


def read(path=OUT):
    """(sha256 recorded, {(config, row): loss})."""
    sha, vals = None, {}
    if not os.path.exists(path):
        return sha, vals
    for line in open(path):
        if line.startswith("# sources_sha256:"):
            sha = line.split(":", 1)[1].strip()
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = (s.strip() for s in line.split("=", 1))
            name, row = k.rsplit(".row", 1)
            vals[(name, int(row))] = float(v)
    return sha, vals


def main(names):
    sha = sources_sha256()
    old_sha, vals = read()
    if old_sha != sha:
        vals = {}
    o = Oracle("f64")
    for name in names:
        cfg = syn.CONFIGS[name]
        params = syn.init_params(cfg).astype(o.dtype)
        tok, tgt = syn.draw_tokens(cfg)
        for b in range(cfg.B):
            if (name, b) in vals:
                continue
            t0 = time.time()
            m = o.model(cfg.dims(), 1, cfg.T)
            vals[(name, b)] = float(m.forward(params, tok[b:b + 1], tgt[b:b + 1]))
            del m
            print(f"{name} row {b}: {vals[(name, b)]!r} ({time.time() - t0:.0f} s)", flush=True)
            write(sha, vals)
    write(sha, vals)


def write(sha, vals):
    lines = ["# Mean cross-entropy over the T positions of each row of the full-size",
             "# workloads (seeded inputs of synthetic.py), from the double-precision",
             "# oracle, one B = 1 forward per row.  Written by make_row_losses.py.",
             f"# sources_sha256: {sha}",
             f"# ({' + '.join(HASHED)})"]
    for name in CONFIGS:
        for (n, b), v in sorted(vals.items(), key=lambda kv: kv[0][1]):
            if n == name:
                lines.append(f"{name}.row{b} = {v!r}")
    tmp = OUT + ".tmp"
    with open(tmp, "w") as f:
        f.write("\n".join(lines) + "\n")
    os.replace(tmp, OUT)


if __name__ == "__main__":
    main(sys.argv[1:] or list(CONFIGS))
