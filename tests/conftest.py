import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libqdecode")
    config.addinivalue_line("markers", "slow: full-size case (minutes on CPU)")


def golden_rows(name):
    """Non-comment, whitespace-split rows of a golden fixture file."""
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


@pytest.fixture(scope="session")
def cuda_ok():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return True


@pytest.fixture(scope="session")
def qd(cuda_ok):
    """The CUDA library's Python binding (fails loudly when the extension is missing)."""
    import quantized_decode_gemv_gb300 as q

    q.load()
    return q
