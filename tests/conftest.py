import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: large seeded workloads (minutes of host time)")


@pytest.fixture(scope="session")
def workloads():
    """Seeded workloads, generated once per session and cached by (id, batch)."""
    import tt_inputs

    cache = {}

    def get(cid, batch=None):
        key = (cid, batch)
        if key not in cache:
            cache[key] = tt_inputs.config(cid, batch=batch)
        return cache[key]

    return get
