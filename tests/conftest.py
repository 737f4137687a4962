import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built extension")


def read_golden(name: str) -> dict:
    """Parse a `key = value` fixture; values are split on whitespace."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = (t.strip() for t in line.split("=", 1))
            out[k] = v.split()
    return out


def as_ints(v):
    return [int(t, 0) for t in v]


def as_floats(v):
    return [float(t) for t in v]


@pytest.fixture(scope="session")
def golden_hand():
    return read_golden("hand_examples.txt")


@pytest.fixture(scope="session")
def golden_facts():
    return read_golden("format_facts.txt")
