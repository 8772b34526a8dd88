import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def qk_lib():
    """The CUDA library, built in-tree if needed (nvcc cross-compiles without a GPU)."""
    from quantized_q4_matmul_gb300 import build as qk_build
    qk_build.build()
    import quantized_q4_matmul_gb300 as qk
    return qk


@pytest.fixture(scope="session")
def cuda(qk_lib):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The achieved max|err| / rms of every parity check of the session, worst
    first (the bar is 1e-2)."""
    try:
        from tests import test_gpu_parity
    except Exception:
        return
    margins = getattr(test_gpu_parity, "MARGINS", [])
    if not margins:
        return
    worst = sorted(margins, key=lambda m: -m[1])
    terminalreporter.write_line("parity margins: %d checks, max|err|/rms worst %.2e, median %.2e (bar 1e-2)" % (
        len(margins), worst[0][1], sorted(m[1] for m in margins)[len(margins) // 2]))
    for what, r in worst[:12]:
        terminalreporter.write_line("  %.2e  %s" % (r, what))
