import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the compiled selector library")
    config.addinivalue_line("markers", "slow: full-size parity case (several seconds of CPU oracle work)")


def pytest_collection_modifyitems(config, items):
    # GPU tests are skipped (not failed) when no GPU is present; the -m filter decides what runs.
    try:
        import torch

        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device in this environment")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """Prints the per-config counts of the full-size oracle comparisons (rows compared,
    near-tie steps) that the GPU parity tests collected."""
    try:
        import parity_rules
    except ImportError:  # pragma: no cover
        return
    if parity_rules.REPORT:
        terminalreporter.section("full-size comparison with the oracle")
        for line in parity_rules.REPORT:
            terminalreporter.write_line(line)
