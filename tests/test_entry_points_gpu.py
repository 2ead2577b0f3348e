"""The entry points the parity tests do not go through: the allocating
ssd_complex_fwd (workspace from cudaMallocAsync on the caller's stream) and the
per-launch timing instrumentation. The allocating call must give the same bits
as the workspace call on the same inputs, and both the oracle's result."""
import numpy as np
import pytest
import torch

from oracle import naive_scan_inputs
from state_space_sequence_complex_gb300 import inputs, ssdc
from tests.gpu_util import assert_close, run_library, to_device

pytestmark = pytest.mark.gpu

ORDER = ["x_re", "x_im", "A_re", "A_im", "B_re", "B_im", "C_re", "C_im", "dt"]


@pytest.fixture(scope="module", autouse=True)
def built():
    from state_space_sequence_complex_gb300 import build
    build.build()
    ssdc.load()


@pytest.mark.parametrize("precision,Q,dims", [("fp32", 32, (2, 200, 3, 16, 16)), ("tf32", 64, (2, 320, 3, 64, 64)),
                                              ("tf32", 128, (1, 300, 2, 64, 64))])
def test_allocating_entry_point(precision, Q, dims):
    inp = inputs.custom(*dims, seed=601 + Q)
    t = to_device(inp)
    y_re, y_im, fs_re, fs_im = ssdc.ssd_complex_fwd(*[t[k] for k in ORDER], Q, precision)
    torch.cuda.synchronize()
    y = y_re.double().cpu().numpy() + 1j * y_im.double().cpu().numpy()
    s = fs_re.double().cpu().numpy() + 1j * fs_im.double().cpu().numpy()
    assert_close(y, s, *naive_scan_inputs(inp), precision, "allocating entry point")
    yw, sw, _ = run_library(inp, Q, precision, dev=t)
    assert np.array_equal(y, yw) and np.array_equal(s, sw)


def test_timing_instrumentation_reports_each_launch():
    inp = inputs.custom(1, 256, 2, 64, 64, seed=611)
    t = to_device(inp)
    for precision, launches in (("tf32", 1), ("tf32_staged", 3), ("fp32", 3)):
        f = ssdc.Forward(*inp.dims, 64, precision)
        ssdc.timing_enable(True)
        try:
            f(*[t[k] for k in ORDER])
            ms = ssdc.timing_read(8)
        finally:
            ssdc.timing_enable(False)
        assert ssdc.last_launch_count() == launches
        assert len(ms) == launches and all(m > 0 for m in ms)
        assert f.status() == ssdc.SSDC_OK
