import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a B300 GPU (sm_103a) and libmg.so")


def load_golden(name):
    """Parse tests/golden/<name>: 'key value rel_tol source...' lines."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            out[parts[0]] = (float(parts[1]), float(parts[2]), " ".join(parts[3:]))
    return out


@pytest.fixture(scope="session")
def golden_bytes():
    return load_golden("kv_bytes.txt")
