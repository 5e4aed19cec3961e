import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def root_dir():
    return ROOT


@pytest.fixture
def kernel_family(request):
    """Indirect parameter: run the test on one kernel family ("tcgen05",
    "mma", "simt"); the automatic choice is restored afterwards."""
    from matrix_state_non_gb300 import binding
    with binding.kernel_family(request.param):
        yield request.param
