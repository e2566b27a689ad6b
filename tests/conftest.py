import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libfattn")
    config.addinivalue_line("markers", "slow: longer CPU test")


@pytest.fixture(scope="session")
def cuda_device():
    import torch

    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    return torch.device("cuda:0")


def pytest_terminal_summary(terminalreporter):
    """One line over every oracle comparison of the run: the largest errors,
    and how many elements needed the wider bar at |O| >= 4 (1e-2 + half a
    bf16 ulp)."""
    try:
        from tests.gpu_helpers import PARITY_LOG
    except ImportError:
        return
    if not PARITY_LOG:
        return
    st = [s for _, s in PARITY_LOG]
    n = sum(s.n_elements for s in st)
    over = sum(s.n_over_1e2 for s in st)
    worst = max(s.worst_over_ulps for s in st)
    terminalreporter.write_line(
        f"parity summary: {len(st)} passing comparisons, {n} output elements; max|dO| {max(s.max_o for s in st):.3e}, "
        f"max mean|dO| {max(s.mean_o for s in st):.3e}, max|dLSE| {max(s.max_l for s in st):.3e}; "
        f"{over} elements over 1e-2 (all at |O| >= 4), worst {worst:.2f} bf16 ulp")
