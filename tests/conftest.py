import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_terminal_summary(terminalreporter):
    """One line per full-size workload comparison with its error margins."""
    try:
        from parity import MARGINS
    except ImportError:
        return
    rows = [m for m in MARGINS if m[0].startswith("workload")]
    if not rows:
        return
    terminalreporter.write_line("parity margins (GPU vs fp64 oracle):")
    f = lambda x: "-" if x is None else f"{x:.3e}"
    for name, eo, mo, es in rows:
        terminalreporter.write_line(f"  {name}: out rel-L2 {f(eo)} max-abs {f(mo)}; state rel-L2 {f(es)}")
