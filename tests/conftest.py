import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


# Lines that tests add (decision and near-tie counts, measured rates); printed
# after the run so that they appear at the end of the log.
SUMMARY = []


def pytest_terminal_summary(terminalreporter):
    if SUMMARY:
        terminalreporter.write_sep("-", "measured counts")
        for line in SUMMARY:
            terminalreporter.write_line(line)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def gpu_available() -> bool:
    try:
        import torch

        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def lib():
    """The built libdspark binding (builds it in-tree on first use)."""
    from draft_sampling_lossless_gb300 import build

    build.ensure_built()
    from draft_sampling_lossless_gb300 import binding

    return binding


def pytest_collection_modifyitems(config, items):
    if gpu_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)
