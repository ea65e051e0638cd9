import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size parity case (seconds to minutes)")


def load_golden(name):
    """Parse a tests/golden/*.txt fixture: '# ...' comments, then 'key v1 v2 ...' lines."""
    path = os.path.join(ROOT, "tests", "golden", name)
    out = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = [int(v) for v in vals]
    return out


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.default()
