import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 and the built CUDA library")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built libkime_attn on a visible GPU (builds it if needed)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from packed_varlen_attention_kime_gb300 import build, load_library
    build.build()
    return load_library()
