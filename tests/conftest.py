import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300); calls the C ABI on the device")


@pytest.fixture(scope="session")
def oracle():
    from oracle import ref_scan
    ref_scan.build()
    return ref_scan


@pytest.fixture(scope="session")
def ssmlib():
    """libssmscan built in-tree (nvcc cross-compiles without a GPU) and loaded."""
    from selective_state_space_fwd_gb300 import build, _binding
    build.build()
    _binding.load()
    return _binding
