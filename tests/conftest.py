import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def kvq_lib_path():
    """Path of the compiled C-ABI library, building it first if it is missing."""
    import __graft_entry__ as ge

    path = ge.library_path()
    if not os.path.exists(path):
        ge.build()
    return path
