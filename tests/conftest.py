import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.lib()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """Worst output element of every GPU parity comparison, as a fraction of the
    tolerance (1.0 = at the tolerance)."""
    try:
        from tests.parity_util import WORST
    except Exception:
        return
    if not WORST:
        return
    terminalreporter.write_sep("-", "parity: worst element / tolerance")
    for key in sorted(WORST):
        terminalreporter.write_line(f"{WORST[key]:.4f}  {key}")
