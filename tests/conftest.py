import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.dirname(os.path.abspath(__file__))
for p in (ROOT, HERE):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300) and the built library")
    config.addinivalue_line("markers", "slow: long-running check")


@pytest.fixture(scope="session")
def orc():
    import oracle

    oracle.build()
    return oracle


def _cuda_ok():
    try:
        import torch

        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _cuda_ok():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """The measured errors of the parity tests: the row-normalised metric the
    tests assert, next to the pages' element-wise metric (relative with a 1e-6
    floor)."""
    try:
        import _gpu
    except Exception:
        return
    if not _gpu.REPORT:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity errors: row-normalised | element-wise (rel, 1e-6 floor)")
    for test, qty, row, elem in _gpu.REPORT:
        tr.write_line(f"{test:60s} {qty:10s} {row:10.3e} {elem:10.3e}")
