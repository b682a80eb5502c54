import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the compiled CUDA library")
    config.addinivalue_line("markers", "slow: full-size parity case (minutes)")


def pytest_collection_modifyitems(config, items):
    # GPU tests cannot run without a device; skip them explicitly rather than
    # letting them fail on a CPU-only machine when selected by accident.
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


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    # the max-abs error every parity check reached, per case and tensor;
    # also written to the file SWA_PARITY_REPORT names, when set
    from tests import helpers

    if not helpers.REPORT:
        return
    lines = helpers.format_report()
    for line in lines:
        terminalreporter.write_line(line)
    path = os.environ.get("SWA_PARITY_REPORT")
    if path:
        with open(path, "w") as f:
            f.write("\n".join(lines) + "\n")
