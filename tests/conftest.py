import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


def golden(name: str) -> dict:
    """Parse a tests/golden/*.txt fixture: ``key = value | citation`` lines."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kv = line.split("|", 1)[0]
            k, v = kv.split("=", 1)
            out[k.strip()] = float(v.strip())
    return out


@pytest.fixture(scope="session")
def page_values():
    return golden("page_values.txt")
