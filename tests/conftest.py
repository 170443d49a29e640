import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a); runs the CUDA library through its C ABI")


@pytest.fixture(scope="session")
def golden_dir():
    return GOLDEN


@pytest.fixture(autouse=True)
def _skip_gpu_tests_without_cuda(request):
    if request.node.get_closest_marker("gpu") is not None:
        import torch
        if not torch.cuda.is_available():
            pytest.skip("needs a CUDA GPU")


@pytest.fixture(scope="session")
def bsf8_lib():
    """The CUDA library, built in-tree for sm_103a if needed."""
    from block_scaled_fp8_weight_gb300 import build, load
    build.build()
    return load()
