import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def repo_root():
    return ROOT


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print the per-case BF16 parity statistics gathered by tests/_tol.py."""
    try:
        import _tol
    except Exception:
        return
    extra = getattr(_tol, "EXTRA", [])
    if not _tol.STATS and not extra:
        return
    tr = terminalreporter
    tr.section("BF16 parity statistics (GPU vs oracle)")
    tr.write_line(f"{'case':58s} {'elements':>9s} {'max ulps':>8s} {'>1 ulp':>7s} {'exact':>7s} "
                  f"{'widened':>8s} {'cap':>6s}")
    for s in _tol.STATS:
        tr.write_line(f"{s['case'][:58]:58s} {s['n']:9d} {s['max_ulps']:8.3f} {s['above_1ulp']:7d} "
                      f"{s['exact_frac']:7.2%} {s['widened_frac']:8.4%} {s['widened_cap']:6.2%}")
    for line in extra:
        tr.write_line(line)
