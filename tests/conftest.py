import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a kernels)")


@pytest.fixture(scope="session")
def orc():
    import oracle

    return oracle.Oracle()


def _cuda_available() -> bool:
    try:
        import torch

        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def uz():
    """The CUDA library binding. Skips only where there is no GPU at all; on a
    GPU machine a missing or broken extension is an error, never a skip."""
    if not _cuda_available():
        pytest.skip("no CUDA device")
    import lossless_bf16_exponent_gb300 as uz

    uz.load()  # raises if libuzip.so is missing
    return uz
