import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def built_lib():
    """The in-tree C library, compiled if it is missing or stale."""
    from weight_only_int4_rtn_gb300 import _build
    return _build.build()


@pytest.fixture(scope="session")
def w4(built_lib):
    """The binding, on a machine with a GPU (GPU tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    import weight_only_int4_rtn_gb300 as w4mod
    w4mod.lib()
    return w4mod
