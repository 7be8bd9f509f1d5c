import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def native_lib():
    """The C-ABI library, (re)built in-tree first if it is missing or older than a source."""
    from top_gating_expert_gb300 import build as b
    b.build_library()
    from top_gating_expert_gb300 import _native
    return _native.lib()
