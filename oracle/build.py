"""Compile the CPU oracle (test infrastructure) into two shared libraries.

``liboracle_f64.so`` computes in double precision and is the parity reference;
``liboracle_f32.so`` is the same source in single precision, the precision the
llm.c CPU trainer runs in, and is what the CPU baseline times.

Flags: -O2 without -ffast-math and with -ffp-contract=off, so every sum is the
plain IEEE sequence the source spells out.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gpt2_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")


def lib_path(precision: str) -> str:
    return os.path.join(OUT_DIR, f"liboracle_{precision}.so")


def build(force: bool = False) -> None:
    os.makedirs(OUT_DIR, exist_ok=True)
    for prec, extra in (("f64", []), ("f32", ["-DORACLE_FLOAT"])):
        out = lib_path(prec)
        if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
            continue
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
               *extra, SRC, "-o", out + ".tmp", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(out + ".tmp", out)


if __name__ == "__main__":
    build(force="--force" in sys.argv)
