import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libk3mla.so")


@pytest.fixture(scope="session")
def gpu_lib():
    """Build (if needed) and load the CUDA library; skip only when no GPU exists."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_latent_attention_k3mla_gb300 import k3mla
    k3mla.load()
    return k3mla
