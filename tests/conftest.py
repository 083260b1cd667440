import json
import math
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a library)")


def _num(v):
    if isinstance(v, str):
        return {"nan": math.nan, "-inf": -math.inf, "inf": math.inf}[v]
    return float(v)


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        d = json.load(f)
    for key in ("logits", "q"):
        if key in d:
            d[key] = np.array([[_num(v) for v in row] for row in d[key]], dtype=np.float32)
    return d


@pytest.fixture(scope="session")
def golden():
    return load_golden
