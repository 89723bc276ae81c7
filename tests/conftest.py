import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libhc.so")


@pytest.fixture(scope="session")
def golden():
    """Values the pages print, keyed by name (tests/golden/pages_printed_values.txt)."""
    path = os.path.join(ROOT, "tests", "golden", "pages_printed_values.txt")
    out = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val, _cite = line.split(None, 2)
            out[key] = float(val)
    return out
