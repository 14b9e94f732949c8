import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU statistics")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def _tally():
    try:
        import gpu_helpers
    except Exception:  # pragma: no cover
        return None
    return gpu_helpers


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Prints the session's stochastic parity tally (excused near-boundary
    differences against verified positions, and the near-flag rate per kind)."""
    h = _tally()
    for line in (h.tally_lines() if h else []):
        terminalreporter.write_line(line)


def pytest_sessionfinish(session, exitstatus):
    """The parity budget holds over the whole session: excused near-boundary
    differences must stay below 1e-4 of all verified positions."""
    h = _tally()
    if not h:
        return
    exc, pos = h.tally_totals()
    if pos and exc >= h.PARITY_BUDGET * pos:
        session.exitstatus = pytest.ExitCode.TESTS_FAILED
        print(f"\nparity budget exceeded: {exc} excused differences in {pos} positions "
              f"(>= {h.PARITY_BUDGET:.0e})")
