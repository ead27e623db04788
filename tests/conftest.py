import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built extension")
    config.addinivalue_line("markers", "slow: long-running CPU check")


@pytest.fixture(scope="session")
def cuda_lib():
    """The loaded C-ABI library on a GPU machine (fails loudly when the build is missing)."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_sparse_head_gb300 as bsa

    return bsa.load_library()


_PARITY_LINES: list[str] = []


@pytest.fixture(scope="session")
def parity_report():
    """Lines of full-size parity figures, printed in the terminal summary."""
    return _PARITY_LINES


def pytest_terminal_summary(terminalreporter):
    if _PARITY_LINES:
        terminalreporter.write_sep("-", "full-size parity against the oracle")
        for line in _PARITY_LINES:
            terminalreporter.write_line(line)
