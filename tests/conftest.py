import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("this test needs a CUDA device; run it with -m gpu on a GPU host")
    return torch.device("cuda", 0)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    try:
        import parity
    except ImportError:
        return
    path = os.environ.get("FA512_PARITY_LOG")
    if path and parity.RECORDS:
        parity.write_log(path)
    for line in parity.summary_lines():
        terminalreporter.write_line(line)
