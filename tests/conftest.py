import os
import sys

import pytest

# deterministic cuBLAS for the reference products some GPU tests take with torch
os.environ.setdefault("CUBLAS_WORKSPACE_CONFIG", ":4096:8")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size parity cases (tens of seconds)")


@pytest.fixture(autouse=True)
def _poison_uninitialised(request):
    """In GPU tests every tensor made by torch.empty / empty_like (outputs,
    saved buffers and workspaces allocated by the binding included) starts as
    NaN (floating point) or all-ones bytes (integers, so 0xFF in the byte
    buffers: NaN when read as fp32 or bf16).  An element the library never
    writes then shows up as a non-finite value in the parity check instead of
    hiding behind whatever a recycled allocation held."""
    if request.node.get_closest_marker("gpu") is None:
        yield
        return
    import torch

    prev_det = torch.are_deterministic_algorithms_enabled()
    prev_warn = torch.is_deterministic_algorithms_warn_only_enabled()
    prev_fill = torch.utils.deterministic.fill_uninitialized_memory
    torch.use_deterministic_algorithms(True, warn_only=True)
    torch.utils.deterministic.fill_uninitialized_memory = True
    try:
        yield
    finally:
        torch.utils.deterministic.fill_uninitialized_memory = prev_fill
        torch.use_deterministic_algorithms(prev_det, warn_only=prev_warn)
