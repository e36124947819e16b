import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workload (minutes of CPU oracle time)")


def pytest_terminal_summary(terminalreporter):
    """Prints the parity counters the tests recorded (rows, elements compared, elements that pass
    only through a tolerance term, admissible near-boundary tokens, ...), one line per entry."""
    try:
        from helpers import PARITY_COUNTS
    except Exception:
        return
    if not PARITY_COUNTS:
        return
    terminalreporter.write_line("parity counts:")
    for key in sorted(PARITY_COUNTS):
        items = ", ".join(f"{k}={v}" for k, v in sorted(PARITY_COUNTS[key].items()))
        terminalreporter.write_line(f"  {key}: {items}")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle
