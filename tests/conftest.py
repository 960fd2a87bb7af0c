import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def load_golden(name):
    """Parse a tests/golden/*.txt fixture into a dict of scalars and float arrays."""
    path = os.path.join(GOLDEN, name)
    out = {}
    key = None
    rows = []
    with open(path) as f:
        lines = [ln.strip() for ln in f if ln.strip() and not ln.lstrip().startswith("#")]

    def flush():
        if key is not None and rows:
            out[key] = np.array(rows, dtype=np.float64)

    for ln in lines:
        parts = ln.split()
        if len(parts) == 2 and parts[0] in ("M", "N", "K", "alpha", "beta"):
            flush()
            key, rows = None, []
            out[parts[0]] = float(parts[1]) if parts[0] in ("alpha", "beta") else int(parts[1])
        elif len(parts) == 1 and parts[0][0].isalpha():
            flush()
            key, rows = parts[0], []
        else:
            rows.append([float(x) for x in parts])
    flush()
    return out


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle

    oracle.build()
    return oracle
