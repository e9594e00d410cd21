import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: long CPU test (exhaustive sweeps)")


@pytest.fixture(scope="session")
def has_gpu():
    import torch
    return torch.cuda.is_available()


def pytest_terminal_summary(terminalreporter):
    """Report the parity counts of the run: codes and scales compared with the
    oracle and the codes that differ by one step inside the 2-ulp window
    (codes outside it, or any scale mismatch, fail their test)."""
    pu = sys.modules.get("parity_util")
    if pu is None or not pu.TOTALS["elements"]:
        return
    t = pu.TOTALS
    terminalreporter.write_line(
        f"parity: {t['elements']} codes and {t['scales']} scales compared with the oracle; "
        f"{t['window_mismatch']} codes differ by one step inside the 2-ulp window "
        "(a code outside it, or any differing scale, fails its test)")
