import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running CPU oracle work")


def read_golden(name):
    """Parse a `key = values` fixture; `;` separates matrix rows."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            rows = [[float(x) for x in r.split()] for r in val.split(";")]
            out[key] = rows[0] if len(rows) == 1 else rows
            if len(rows) == 1 and len(rows[0]) == 1:
                out[key] = rows[0][0]
    return out


@pytest.fixture
def golden():
    return read_golden
