import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a); runs the CUDA path through the C ABI")


@pytest.fixture(scope="session", autouse=True)
def _built_host_libs():
    """Builds the generator and the oracle once per session (plain gcc, seconds)."""
    import oracle
    import synth
    if not os.path.exists(synth._HOST_LIB):
        synth.lib()
    oracle.build()
    yield
