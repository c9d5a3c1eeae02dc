"""Shared pytest configuration.

Markers:
  gpu -- needs a CUDA device (GB300, sm_103a) and the built library; the CPU
         suite runs with ``-m "not gpu"``.
"""
import os
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

GOLDEN = Path(__file__).resolve().parent / "golden"


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: test needs a CUDA GPU and the built library")


@pytest.fixture(scope="session")
def golden_dir():
    return GOLDEN
