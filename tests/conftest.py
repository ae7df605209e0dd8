import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long CPU test")


def pytest_collection_modifyitems(config, items):
    # GPU tests fail loudly (not skip) when the GPU or the library is missing;
    # they are selected with -m gpu only where a GPU exists.
    pass


@pytest.fixture(scope="session")
def oracle():
    import oracle as o
    o.lib()
    return o


@pytest.fixture(scope="session")
def W():
    """The CUDA library's binding, built for sm_103a; a GPU must be present."""
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from w8a8_gemm_rl_gb300 import _build
    _build.build()
    import w8a8_gemm_rl_gb300 as w
    w.lib()
    return w
