import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def load_golden(name):
    """Read a text fixture under tests/golden: blocks of 'name rows cols'
    followed by one line of row-major values."""
    import numpy as np
    path = os.path.join(ROOT, "tests", "golden", name)
    out = {}
    lines = [l.strip() for l in open(path) if l.strip() and not l.startswith("#")]
    for i in range(0, len(lines), 2):
        key, r, c = lines[i].split()
        vals = [float(v) for v in lines[i + 1].split()]
        out[key] = np.array(vals, dtype=np.float64).reshape(int(r), int(c))
    return out
