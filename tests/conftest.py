import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libfp4.so")


def read_golden(name):
    """Parse a tests/golden text fixture: '#' comments, 'key = values' lines
    or plain whitespace-separated rows."""
    kv, rows = {}, []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if "=" in line:
                k, v = line.split("=", 1)
                kv[k.strip()] = v.split()
            else:
                rows.append(line.split())
    return kv, rows


@pytest.fixture(scope="session")
def O():
    import oracle
    oracle.lib()
    return oracle
