import os, sys
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
"""Test configuration: the `gpu` marker and shared fixtures.

CPU tests (``-m "not gpu"``) pin the oracle and check the host-side logic and
the library's exported symbols.  GPU tests (``-m gpu``) compare the CUDA path
with the oracle through the C ABI.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300 / sm_103a)")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.lib()
    return oracle


def _cuda_ok():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def kvq():
    """The CUDA library binding; GPU tests fail (not skip) if it cannot load."""
    if not _cuda_ok():
        pytest.skip("no CUDA device")
    from fp8_paged_kv_attn_gb300 import kvq as binding
    binding.load()
    return binding
