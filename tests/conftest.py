"""Shared pytest configuration.

``-m gpu`` tests call the CUDA library through its C ABI on a GPU; everything
else runs on the CPU (oracle pins, host-side validation, symbol exports,
the replica launcher under gloo).
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size parity cases (seconds to a minute each)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built CUDA library, loaded through the Python binding (GPU tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from confidence_driven_speculative_gb300 import binding
    binding.load()
    return binding
