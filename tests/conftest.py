import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: CPU test that takes more than a few seconds")


def has_cuda() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def gpt_lib():
    """The built CUDA library through its binding; a GPU test without it fails loudly."""
    if not has_cuda():
        pytest.fail("gpu test selected but no CUDA device is visible")
    from decoder_only_transformer_gpt_gb300 import binding
    return binding.load()
