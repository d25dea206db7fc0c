import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def built_lib():
    """Builds libncc_gb300.so in-tree if it is missing or stale."""
    from normalized_cross_correlation_gb300 import _build
    return _build.build()


@pytest.fixture(scope="session")
def ncc(built_lib):
    """The Python binding, for tests that run kernels (GPU only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from normalized_cross_correlation_gb300 import ncc as binding
    binding.lib()
    return binding


@pytest.fixture(scope="session")
def threads():
    import oracle
    return oracle.default_threads()
