import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


@pytest.hookimpl(tryfirst=True)
def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-shape case (minutes of CPU oracle work)")
    # every test is bounded (pytest-timeout, where installed; an explicit --timeout wins): a test
    # stuck on a kernel that does not return ends, dumping its stack, instead of holding the GPU
    if config.pluginmanager.hasplugin("timeout") and not getattr(config.option, "timeout", None):
        config.option.timeout = 900
        config.option.timeout_method = "thread"


@pytest.fixture(scope="session")
def cuda_lib():
    """The built C-ABI library; GPU tests fail (not skip) when it is missing."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    from deepseek_v4_moe_gb300 import _lib
    return _lib.load()
