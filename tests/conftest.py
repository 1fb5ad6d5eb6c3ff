import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def golden(name: str) -> dict:
    """Parse a tests/golden fixture: 'key: value' lines, '#' comments."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = line.split(":", 1)
            vals = val.split()
            out[key.strip()] = [float(x) for x in vals] if len(vals) > 1 else float(vals[0])
    return out


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle
