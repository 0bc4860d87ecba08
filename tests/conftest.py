import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libselscan")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes of host time)")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle._load()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """The worst forward parity figures of the session: relative L2, the condition-aware max
    relative error (fp32) and the plain max |e| / max |y_ref|, per I/O type."""
    try:
        from helpers import RECORDED
    except ImportError:
        return
    if not RECORDED:
        return
    tr = terminalreporter
    tr.write_sep("-", "forward parity against the oracle (worst case over the session)")
    for io in ("f32", "bf16"):
        rows = [r for r in RECORDED if r[1] == io]
        if not rows:
            continue
        worst_l2 = max(rows, key=lambda r: r[2])
        worst_pm = max(rows, key=lambda r: r[4])
        line = (f"{io}: {len(rows)} checks; rel-L2 {worst_l2[2]:.3e} ({worst_l2[0]}); "
                f"plain max|e|/max|y| {worst_pm[4]:.3e} ({worst_pm[0]})")
        if io == "f32":
            worst_mr = max(rows, key=lambda r: r[3])
            line += f"; max-rel {worst_mr[3]:.3e} ({worst_mr[0]})"
        tr.write_line(line)
