import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def golden_path(name):
    return os.path.join(ROOT, "tests", "golden", name)


def read_golden(name):
    """key = value lines; '#' starts a comment."""
    vals = {}
    with open(golden_path(name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            vals[key] = val
    return vals


@pytest.fixture(scope="session")
def pool():
    """A spawn-started process pool that runs the oracle on full-size
    batches (tests/oracle_pool.py)."""
    from oracle_pool import OraclePool
    p = OraclePool()
    yield p
    p.close()
