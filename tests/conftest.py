import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA library through its C ABI)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library through its Python binding; skips only when no GPU exists.

    On a machine with a GPU a missing or unbuildable library is an error, never a skip.
    """
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device on this machine")
    import ggml_quantized_dequant_gb300 as qdq
    qdq.load()  # raises if the shared library is missing
    return qdq
