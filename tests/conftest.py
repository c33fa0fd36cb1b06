import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libgdn.so")


@pytest.fixture(autouse=True)
def _no_oracle_mutation():
    """Every test starts and ends with the oracle unmutated."""
    try:
        import oracle
    except Exception:  # pragma: no cover
        yield
        return
    oracle.set_mutation(0)
    yield
    oracle.set_mutation(0)
