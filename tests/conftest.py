import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def read_golden(name):
    """Parse a golden fixture: '#' comments, then rows '<tag> <numbers...>'."""
    rows = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            tag, *vals = line.split()
            rows.setdefault(tag, []).append([float(v) for v in vals])
    return {k: np.array(v, dtype=np.float64) for k, v in rows.items()}


@pytest.fixture(scope="session")
def golden():
    return read_golden
