"""Test configuration.

Markers: ``gpu`` -- needs a CUDA device (GB300, sm_103a) and the built
library; everything else runs on a CPU-only machine.
"""
from __future__ import annotations

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def cuda_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def zlib():
    """The C-ABI library, built in-tree if it is missing or stale."""
    import zero_sharded_mixed_shard_gb300 as z
    z.build()
    return z
