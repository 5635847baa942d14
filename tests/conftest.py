import os
import sys
from fractions import Fraction
import math

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def _parse_value(tok: str) -> float:
    if tok == "L3":
        return math.log(3.0)
    if "/" in tok:
        return float(Fraction(tok))
    return float(tok)


def load_golden(name: str) -> dict:
    """Parse a golden text fixture: '<key> v1 v2 ...' lines, '#' comments.
    Returns key -> 2-D float64 array (one row per line with that key)."""
    rows: dict = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            rows.setdefault(key, []).append([_parse_value(v) for v in vals])
    return {k: np.array(v, dtype=np.float64) for k, v in rows.items()}


@pytest.fixture
def golden():
    return load_golden
