import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes)")


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _has_gpu():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print how many GEMM outputs each parity check accepted only through the
    near-tie rule (the BF16 neighbour across a rounding boundary)."""
    from tests.helpers import TIE_LOG
    if not TIE_LOG:
        return
    tr = terminalreporter
    tr.write_sep("-", "GEMM near-tie acceptances (outputs checked / accepted by the near-tie rule)")
    total = checked = 0
    for label, n, ties in TIE_LOG:
        tr.write_line(f"{ties:>8d} / {n:<10d} {label}")
        total += ties
        checked += n
    tr.write_line(f"{total:>8d} / {checked:<10d} all checks ({(total / checked if checked else 0.0):.5%})")
