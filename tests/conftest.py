import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device of compute capability 10.3 (sm_103)")
    config.addinivalue_line("markers", "slow: large-size case (minutes)")


@pytest.fixture(scope="session")
def lib():
    """The built C-ABI library (built on demand; CPU machines can load it too)."""
    from co_folding_pair_gb300 import _lib
    return _lib.load()


def pytest_terminal_summary(terminalreporter):
    from tests._util import RECORD
    if not RECORD:
        return
    terminalreporter.section("parity against the fp64 oracle")
    for what, worst, fro in RECORD:
        terminalreporter.write_line(f"{what:40s} worst element {worst:.3f} of bound, rel Frobenius {fro:.2e}")
