import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a); parity tests proper")
    config.addinivalue_line("markers", "slow: large-shape parity case")


@pytest.fixture(autouse=True)
def _require_cuda_for_gpu_tests(request):
    if request.node.get_closest_marker("gpu") is not None:
        import torch
        if not torch.cuda.is_available():
            pytest.skip("no CUDA device in this process")


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
