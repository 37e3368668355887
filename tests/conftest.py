import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def read_golden(name):
    """Parse a tests/golden/*.txt fixture: '# comments', 'key v1 v2 ...'."""
    path = os.path.join(ROOT, "tests", "golden", name)
    out = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            vals = [float(x) for x in vals]
            if key in out:
                if not isinstance(out[key][0], list):
                    out[key] = [out[key]]
                out[key].append(vals)
            else:
                out[key] = vals
    return out


@pytest.fixture
def golden():
    return read_golden
