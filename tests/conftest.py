"""Shared pytest configuration.

GPU tests carry ``@pytest.mark.gpu``; everything else runs on a CPU-only
machine.  The repository root is put on sys.path so that ``oracle``,
``workloads`` and the library package import without installation.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a)")
