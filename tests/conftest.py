import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built GPU library")
    config.addinivalue_line("markers", "slow: full-size workload (minutes)")


def read_golden(name):
    """Parse a golden fixture: 'key v1 v2 ...' lines, '#' comments.  Values kept as strings."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, *vals = line.split()
                out[key] = vals
    return out
