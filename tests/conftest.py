import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: longer CPU test")


@pytest.fixture(scope="session")
def golden():
    import json

    def load(name):
        with open(os.path.join(GOLDEN, name)) as f:
            return json.load(f)

    return load


def pytest_terminal_summary(terminalreporter):
    """Decision and near-tie counts of the GPU parity tests, printed under -q too."""
    from tests._parity import RECORD
    if not RECORD:
        return
    terminalreporter.write_sep("-", "parity: decisions and near-ties (|u - p/q| < 1e-6 or "
                                    "Gumbel top-2 gap < 1e-6, on the oracle's values)")
    for what, dec, near, near_o in RECORD:
        terminalreporter.write_line(f"{what}: {dec} decisions, {near} differing at a near-tie, "
                                    f"{near_o} near-ties in the oracle's round")
