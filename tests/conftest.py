import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workload checks (minutes)")


@pytest.fixture(scope="session", autouse=True)
def _host_libs():
    """Compile the C generator and the C oracle once per session (gcc, seconds)."""
    import oracle
    import synth
    synth.build()
    oracle.build()
    yield
