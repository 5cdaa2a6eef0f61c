import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (runs the sm_103a library)")


@pytest.fixture(scope="session")
def gpu_lib():
    """Build (if stale) and load the CUDA library; a GPU test fails loudly without it."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("this test needs a CUDA device")
    from mla_latent_kv_08_gb300 import build as _build
    _build.build()
    import mla_latent_kv_08_gb300 as mla
    return mla.load_library()
