import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Near ties and ambiguous substitutions excluded from the bit-exact
    comparisons, per test case (the parity rule asks for the count)."""
    try:
        from parity import TIES
    except Exception:  # pragma: no cover
        return
    if not TIES:
        return
    tr = terminalreporter
    tr.section("excluded from bit-exact comparison (near ties within 1e-6)")
    for key, (n, total) in TIES.items():
        tr.write_line(f"{key}: {n} of {total}")
