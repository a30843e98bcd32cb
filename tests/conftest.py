import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libgsa.so")
    config.addinivalue_line("markers", "slow: full-size workload (minutes)")


def read_golden(name):
    """Rows of whitespace-separated fields from tests/golden/<name>, comments dropped."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def parse_num(s):
    return int(s, 16) if s.lower().startswith(("0x", "-0x")) else float(s)
