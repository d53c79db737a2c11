import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU case")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Per-case attention errors against the oracle: the mean error over the
    bf16-rounding floor and the worst element over its bound."""
    try:
        import parity_bar
    except ImportError:
        return
    lines = parity_bar.summary_lines()
    if lines:
        terminalreporter.write_sep("-", "attention parity vs the fp64 oracle (bf16 floor)")
        for ln in lines:
            terminalreporter.write_line(ln)
