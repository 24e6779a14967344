import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libtq.so")
    config.addinivalue_line("markers", "slow: longer CPU test")


@pytest.fixture(scope="session")
def root():
    return ROOT


@pytest.fixture(scope="session")
def tqlib():
    """Builds (if needed) and loads libtq.so; the package itself never falls back."""
    from turboquant_quantized_kv_gb300 import build as tqbuild
    tqbuild.build()
    import turboquant_quantized_kv_gb300 as tq
    tq.lib()
    return tq


@pytest.fixture(scope="session")
def cuda(tqlib):
    import torch
    if not torch.cuda.is_available():
        raise RuntimeError("GPU tests need a CUDA device")
    torch.cuda.init()
    return torch
