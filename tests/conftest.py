import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running (large workloads)")


def load_golden(name):
    """Parse a tests/golden/*.txt fixture: '#' comments, 'key value' scalars,
    and 'key' followed by rows of numbers (a matrix)."""
    scalars, mats, cur = {}, {}, None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            try:
                row = [float(p) for p in parts]
            except ValueError:
                row = None
            if row is not None and cur is not None:
                mats[cur].append(row)
            elif len(parts) == 2 and row is None and _isnum(parts[1]):
                scalars[parts[0]] = float(parts[1])
                cur = None
            else:
                cur = parts[0]
                mats[cur] = []
    out = {k: np.array(v, dtype=np.float64) for k, v in mats.items()}
    out.update(scalars)
    return out


def _isnum(s):
    try:
        float(s)
        return True
    except ValueError:
        return False


def rel_err(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))
