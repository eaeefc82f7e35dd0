import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads")


def pytest_terminal_summary(terminalreporter):
    """The correctly rounded fraction of the 16-bit outputs the GPU tests
    compared (smallest over all, and every check of more than a million
    outputs), so a run's log reports it even when every check passed."""
    try:
        import _parity
    except ImportError:
        return
    log = _parity.CR_LOG
    if not log:
        return
    tr = terminalreporter
    tr.section("correctly rounded 16-bit outputs")
    worst = min(log, key=lambda e: e[2])
    total = sum(e[1] for e in log)
    tr.write_line(f"{len(log)} checks, {total} outputs; smallest fraction {worst[2]:.6f} "
                  f"({worst[0]}, {worst[1]} outputs, {worst[3]} above / {worst[4]} below)")
    for what, n, frac, up, down in log:
        if n >= 1_000_000:
            tr.write_line(f"  {frac:.6f}  {n:>11d}  +{up}/-{down}  {what}")
