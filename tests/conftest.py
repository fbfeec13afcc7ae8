"""Shared pytest set-up: repo root on sys.path and the ``gpu`` marker.

Tests marked ``gpu`` need a CUDA device and the compiled library; everything
else runs on a CPU-only machine.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the compiled CUDA library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


@pytest.fixture(scope="session")
def ssd():
    """The Python binding with libssdscan.so loaded (GPU tests)."""
    from mamba_ssd_selective_gb300 import binding
    binding.load()
    return binding
