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


def pytest_terminal_summary(terminalreporter):
    """Print the worst-case figures the whole-tensor parity checks recorded."""
    mod = sys.modules.get("gpu_util")
    rows = getattr(mod, "PARITY_REPORT", None) if mod else None
    if not rows:
        return
    terminalreporter.write_sep("-", "parity: worst case over every element, against the oracle")
    for what, fields in rows:
        terminalreporter.write_line(
            f"{what}: " + ", ".join(f"{k}={v:.3g}" if isinstance(v, float) else f"{k}={v}"
                                   for k, v in fields.items()))
