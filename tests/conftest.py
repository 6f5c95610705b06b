import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def pytest_terminal_summary(terminalreporter):
    """The parity checks closest to their error bound (largest |err| / bound)."""
    try:
        from tests._helpers import RATIOS
    except ImportError:
        return
    if not RATIOS:
        return
    worst = sorted(RATIOS, reverse=True)[:12]
    terminalreporter.write_line(f"parity: {len(RATIOS)} checks, largest |err|/bound:")
    for r, name in worst:
        terminalreporter.write_line(f"  {r:.4f}  {name}")
