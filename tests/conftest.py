import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def gpu():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The attention parity checks' worst errors: per head (the asserted
    tolerance) and per single row (reported)."""
    rk = sys.modules.get("roundkit")
    if rk is None or not getattr(rk, "ERROR_LOG", None):
        return
    log = rk.ERROR_LOG
    tr = terminalreporter
    tr.section("attention parity: worst errors (tolerance per head: rel-L2 1e-3, max abs 4e-3)")
    tr.write_line(f"checks: {len(log)}")
    for key, name in ((1, "head rel-L2"), (2, "head max-abs"), (3, "row rel-L2"), (4, "row max-abs")):
        worst = max(log, key=lambda e: e[key])
        tr.write_line(f"  worst {name:12s} {worst[key]:.3e}  ({worst[0]})")
