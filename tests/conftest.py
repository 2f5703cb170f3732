import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the compiled library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """The parity exceptions counted during the run (near-ties, accept
    margins and top-p boundaries the comparison excused), one line per check,
    so that a run's log shows how many there were and how close they came."""
    parity = sys.modules.get("parity")
    if parity is None or not parity.EXCEPTIONS:
        return
    tr = terminalreporter
    tot_e = sum(r["exceptions"] for r in parity.EXCEPTIONS)
    tot_n = sum(r["total"] for r in parity.EXCEPTIONS)
    tr.write_sep("=", f"parity exceptions: {tot_e} in {tot_n} compared "
                      f"({len(parity.EXCEPTIONS)} checks)")
    for r in parity.EXCEPTIONS:
        if r["exceptions"] == 0:
            continue
        tr.write_line(f"{r['exceptions']:4d} / {r['total']:<6d} {r['kind']:<52s} smallest "
                      f"{r['smallest']:.3g}  {r['test']}")
    if tot_e == 0:
        tr.write_line("none: every token, accept count and resampled token matched the oracle")
