import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))
for _p in (ROOT, TESTS):
    if _p not in sys.path:
        sys.path.insert(0, _p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_terminal_summary(terminalreporter):
    """Worst parity margins of the run (fractions of the stated bounds)."""
    try:
        from parity import MARGINS
    except ImportError:
        return
    if not MARGINS:
        return
    tr = terminalreporter
    tr.write_sep("-", f"parity margins: {len(MARGINS)} checks (error as a fraction of each bound)")
    worst_rel = max(MARGINS, key=lambda m: m[1])
    worst_elem = max(MARGINS, key=lambda m: m[2])
    tr.write_line(f"worst relative Frobenius: {worst_rel[1]:.3f} of 5e-3 ({worst_rel[0]})")
    tr.write_line(f"worst element: {worst_elem[2]:.3f} of 1e-2 (|ref| + rms) ({worst_elem[0]})")
    for name, rel, elem in sorted(MARGINS, key=lambda m: -m[2])[:12]:
        tr.write_line(f"  {name}: frobenius {rel:.3f}, element {elem:.3f}")
