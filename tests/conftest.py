import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")


def load_golden(name):
    """Parse a `key = value  # citation` fixture from tests/golden/."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            out[key] = val
    return out


def load_worked_9x9():
    """(A, B) as lists of int rows from the worked-example fixture."""
    mats, cur = {}, None
    with open(os.path.join(ROOT, "tests", "golden", "worked_9x9_inputs.txt")) as f:
        for line in f:
            s = line.strip()
            if not s or s.startswith("#"):
                continue
            if s in ("A", "B"):
                cur = s
                mats[cur] = []
                continue
            mats[cur].append([int(v) for v in s.split()])
    return mats["A"], mats["B"]
