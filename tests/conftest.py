import os
import sys

import pytest

ROOT = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(ROOT)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# Worst |y - y_ref| / bound of the tolerance-bounded parity checks of this session, per check:
# the accuracy each one had to spare, printed at the end of the run so that a regression shows
# before it crosses the bound.
WORST = {}


def record_worst(name: str, worst: float) -> None:
    WORST[name] = max(float(worst), WORST.get(name, 0.0))


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_terminal_summary(terminalreporter):
    if not WORST:
        return
    items = sorted(WORST.items(), key=lambda kv: -kv[1])
    terminalreporter.write_sep("-", "worst error / bound of the tolerance-bounded parity checks")
    terminalreporter.write_line(f"{len(items)} checks; the largest ratios:")
    for name, w in items[:12]:
        terminalreporter.write_line(f"  {w:.4f}  {name}")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle
