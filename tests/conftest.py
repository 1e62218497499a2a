import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libdllm.so")


@pytest.fixture(scope="session")
def dllm():
    """The Python binding of libdllm.so, on a GPU.  Fails loudly when the
    library or the GPU is missing (no fallback path exists)."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("gpu test collected without a CUDA device")
    import denoise_step_token_gb300 as pkg
    return pkg


def golden(name):
    import json
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return json.load(f)
