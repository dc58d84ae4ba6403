import os
import sys

import pytest

ROOT = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(ROOT)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libswa.so")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def pytest_terminal_summary(terminalreporter):
    """Whole-output parity figures of the full-size comparisons that ran (shown with -q too)."""
    import parity

    if not parity.RECORDS:
        return
    tr = terminalreporter
    tr.section("whole-output parity against the fp64 oracle")
    tr.write_line(f"{'output':<44} {'rows':>9} {'O elements':>12} {'O max-abs':>10} {'O mean-abs':>10} "
                  f"{'lse max-abs':>11}")
    for what, rows, n_el, mx, mean, lmx in parity.RECORDS:
        tr.write_line(f"{what:<44} {rows:>9} {n_el:>12} {mx:>10.3e} {mean:>10.3e} {lmx:>11.3e}")
