import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def read_golden(name):
    """Parse a ``name value`` golden file (``#`` comments)."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split()
                out[k] = int(v, 0)
    return out


def read_golden_list(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [int(l.split("#", 1)[0].strip(), 0) for l in f if l.split("#", 1)[0].strip()]
