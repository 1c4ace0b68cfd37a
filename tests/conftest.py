"""Test configuration: markers and import paths.

``-m "not gpu"`` runs on any machine (oracle pins, generator, host-side ABI
checks, multi-rank host logic on gloo); ``-m gpu`` runs the CUDA parity tests
through the C-ABI library on ``cuda:0``.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))
for p in (ROOT, TESTS):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
