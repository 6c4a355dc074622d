import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU oracle work")


def read_golden(name):
    """Parse `key = value` lines of a golden file (comments after '#')."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            out[k] = float(v) if any(ch in v for ch in ".e") else int(v)
    return out


@pytest.fixture(scope="session")
def o64():
    from oracle import Oracle
    return Oracle("f64")


@pytest.fixture(scope="session")
def o32():
    from oracle import Oracle
    return Oracle("f32")


def gpu_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False
