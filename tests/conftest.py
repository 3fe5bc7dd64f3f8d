import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built extension")
    config.addinivalue_line("markers", "slow: full-size parity case (minutes)")


@pytest.fixture(scope="session")
def fckl():
    """The product binding, built and loaded; skips nothing: a missing build fails."""
    import chunked_kl_loss_gb300 as m
    m.load()
    return m
