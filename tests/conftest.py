import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a library)")
    config.addinivalue_line("markers", "slow: long CPU oracle runs at full model size")


@pytest.fixture(scope="session", autouse=True)
def _built():
    """Compile whatever is missing or stale (host parts always, CUDA parts when nvcc exists)."""
    import __graft_entry__ as g
    g.build(import_package=False)
    yield
