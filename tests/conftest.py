import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the CUDA library")
    config.addinivalue_line("markers", "slow: full-size case (minutes of oracle time)")


@pytest.fixture(scope="session")
def ref():
    import oracle
    oracle.lib()
    return oracle


@pytest.fixture(scope="session")
def dev():
    """The CUDA library on cuda:0. GPU tests fail (never skip) without it."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("gpu test selected but no CUDA device is visible")
    from combine_fp8_quant_gb300 import build
    build.build()
    import combine_fp8_quant_gb300 as mp
    mp.load()
    return mp
