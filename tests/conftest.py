import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a kernels)")
    config.addinivalue_line("markers", "slow: full-size workload checks")


@pytest.fixture(scope="session", autouse=True)
def _host_libs():
    """Compile the host-side libraries (generator, oracle) once per session."""
    import oracle
    import synth
    synth.build()
    oracle.build()
