import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Achieved parity errors of the workload tests (norm-wise max relative error per
    tensor, and the max abs error where recorded), so that precision changes inside the
    gates stay visible in the test log."""
    try:
        import parity_util
    except ImportError:
        return
    if not parity_util.RECORDED:
        return
    tr = terminalreporter
    tr.section("achieved parity errors (rel = max|gpu - oracle| / max|oracle|)")
    for name, dtype, errs, abs_errs in parity_util.RECORDED:
        if not name.startswith(("c1_", "c2_", "c3_", "c4_", "c5_")):
            continue
        parts = []
        for k, v in errs.items():
            a = abs_errs.get(k)
            parts.append(f"{k} {v:.2e}" + (f" (abs {a:.2e})" if a is not None else ""))
        tr.write_line(f"{name} [{dtype}]: " + ", ".join(parts))
