import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle

    return oracle.load()


@pytest.fixture(scope="session")
def la():
    """The CUDA library's Python binding, built in-tree if needed."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_linear_attention_map_b300 import build as _build

    _build.build()
    import causal_linear_attention_map_b300 as la

    la.load()
    return la
