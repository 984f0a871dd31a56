import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a kernels)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle

    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def golden():
    import json

    def load(name):
        with open(os.path.join(ROOT, "tests", "golden", name)) as f:
            return json.load(f)

    return load


def pytest_terminal_summary(terminalreporter):
    """Every parity report checked in this session: decisions, low-margin and
    excused counts, the largest alpha / probability errors and the excused rows."""
    try:
        from tests.parity import REPORTS
    except Exception:
        return
    if not REPORTS:
        return
    terminalreporter.section("parity reports")
    for name, text in REPORTS:
        terminalreporter.write_line(f"{name}: {text}")
