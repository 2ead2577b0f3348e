import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


@pytest.fixture
def lib_option():
    """Set process-wide library options (ssd_complex_set_option) for one test;
    every option set is put back to its default afterwards."""
    from state_space_sequence_complex_gb300 import ssdc
    touched = set()

    def setter(key, value):
        ssdc.set_option(key, int(value))
        touched.add(key)
    yield setter
    for k in touched:
        ssdc.set_option(k, ssdc.option.DEFAULTS[k])


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Every parity comparison's relative Frobenius errors, and the largest per
    precision (the margin against the tolerance)."""
    try:
        from tests.gpu_util import RECORDED, TOL
    except Exception:
        return
    if not RECORDED:
        return
    tr = terminalreporter
    tr.section("parity errors (relative Frobenius, y and final state)")
    for test, precision, what, ey, es in RECORDED:
        tr.write_line(f"{precision:12s} y {ey:.3e}  state {es:.3e}  {test} {what}")
    for precision in sorted({r[1] for r in RECORDED}):
        rows = [r for r in RECORDED if r[1] == precision]
        my, ms = max(r[3] for r in rows), max(r[4] for r in rows)
        bar = f"(tolerance {TOL[precision]:g})" if precision in TOL else "(recorded, not a parity bar)"
        tr.write_line(f"max {precision}: y {my:.3e}  state {ms:.3e}  over {len(rows)} comparisons {bar}")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300) and the built libssdc.so")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes)")
