import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the CUDA library")


def read_golden(name):
    """Parse a `key = values` fixture; '#' starts a comment line.  Lines without '='
    are returned as rows of whitespace-separated fields under the key None."""
    out = {None: []}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if "=" in line:
                k, v = line.split("=", 1)
                out[k.strip()] = v.split()
            else:
                out[None].append(line.split())
    return out


@pytest.fixture(scope="session")
def ora():
    import oracle
    oracle._load()
    return oracle
