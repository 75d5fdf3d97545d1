import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


_cache = {}


@pytest.fixture(scope="session")
def inputs_of():
    """Seeded host inputs per workload name, generated once per session."""
    import workloads as W

    def get(name):
        if name not in _cache:
            _cache[name] = W.make_inputs(W.WORKLOADS[name])
        return _cache[name]
    return get
