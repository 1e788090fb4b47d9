"""Test configuration: the ``gpu`` marker and import paths.

Tests marked ``gpu`` need a CUDA device and the CUDA library built for it;
everything else runs on a CPU-only machine.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")
