"""The entry point that allocates nothing (ssd_complex_fwd_noalloc).

Callers that cannot allocate device memory while they run the scan (code
inside a memory-pool or allocator hook, latency-critical paths that forbid
allocator calls, embedders with a fixed memory budget) use this variant: the
staged path with its workspace in the library's static device array. These
checks call it through the C ABI on two different problems in a row (the array
keeps the previous call's contents) and compare it with the oracle, within the
path's tolerance, and with ssd_complex_fwd_ws on the same inputs: bit for bit
on the exact path, where both run the same kernels, and within the tolerance
on the staged TF32 path. The device status of every call is read back through
ssd_complex_noalloc_status. This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from oracle import naive_scan_inputs
from state_space_sequence_complex_gb300 import inputs, ssdc
from tests.gpu_util import TOL, rel_fro, to_device

pytestmark = pytest.mark.gpu

ORDER = ["x_re", "x_im", "A_re", "A_im", "B_re", "B_im", "C_re", "C_im", "dt"]


@pytest.fixture(scope="module", autouse=True)
def built():
    from state_space_sequence_complex_gb300 import build
    build.build()
    ssdc.load()


def run_noalloc(inp, Q, precision):
    d = to_device(inp)
    Bn, T, H, N, D = inp.dims
    f32 = dict(dtype=torch.float32, device="cuda")
    out = dict(y_re=torch.empty((Bn, T, H, D), **f32), y_im=torch.empty((Bn, T, H, D), **f32),
               fs_re=torch.empty((Bn, H, N, D), **f32), fs_im=torch.empty((Bn, H, N, D), **f32))
    ssdc.ssd_complex_fwd_noalloc(*[d[k] for k in ORDER], Q, precision=precision, **out)
    assert ssdc.ssd_complex_noalloc_status() == ssdc.SSDC_OK
    y = out["y_re"].double().cpu().numpy() + 1j * out["y_im"].double().cpu().numpy()
    s = out["fs_re"].double().cpu().numpy() + 1j * out["fs_im"].double().cpu().numpy()
    return y, s


def run_ws(inp, Q, precision):
    d = to_device(inp)
    f = ssdc.Forward(*inp.dims, Q, precision)
    y_re, y_im, fs_re, fs_im = f(*[d[k] for k in ORDER])
    torch.cuda.synchronize()
    assert f.status() == ssdc.SSDC_OK
    y = y_re.double().cpu().numpy() + 1j * y_im.double().cpu().numpy()
    s = fs_re.double().cpu().numpy() + 1j * fs_im.double().cpu().numpy()
    return y, s


@pytest.mark.parametrize("precision", ["fp32", "tf32_staged"])
def test_noalloc_matches_workspace_entry_point_twice(precision):
    # two different problems in a row: the second must not see the first's states
    cases = [inputs.custom(2, 700, 4, 64, 64, seed=91), inputs.custom(1, 1000, 3, 64, 64, seed=92)]
    for inp in cases:
        y, s = run_noalloc(inp, 64, precision)
        y_ws, s_ws = run_ws(inp, 64, precision)
        y_ref, s_ref = naive_scan_inputs(inp)
        assert np.all(np.isfinite(y)) and np.all(np.isfinite(s))
        assert rel_fro(y, y_ref) <= TOL[precision] and rel_fro(s, s_ref) <= TOL[precision]
        if precision == "fp32":
            # the same kernels on the same inputs: any stale scratch would show
            assert np.array_equal(y, y_ws) and np.array_equal(s, s_ws)
        else:
            assert rel_fro(y, y_ws) <= TOL[precision] and rel_fro(s, s_ws) <= TOL[precision]


def test_noalloc_rejects_problems_beyond_its_scratch():
    # 2 x 16 heads x 33 chunks of 32 KB states exceed the static buffer
    d = ssdc.dims(2, 64 * 33, 16, 64, 64, "fp32")
    assert ssdc.ssd_complex_fwd_workspace_bytes(d, 64) > ssdc.NOALLOC_SCRATCH_BYTES
    lib = ssdc.load()
    t = torch.empty(16, dtype=torch.float32, device="cuda")
    cin = ssdc.ssdc_cin(t.data_ptr(), t.data_ptr() + 16)
    cout = ssdc.ssdc_cout(t.data_ptr() + 32, t.data_ptr() + 48)
    rc = lib.ssd_complex_fwd_noalloc(cin, cin, cin, cin, t.data_ptr(), d, 64, cout, cout, None)
    assert rc == ssdc.SSDC_ERR_TOO_LARGE
    assert "static" in ssdc.strerror(rc)
    # the fused path has no scratch to hold: not offered here
    d2 = ssdc.dims(1, 128, 2, 64, 64, "tf32")
    assert lib.ssd_complex_fwd_noalloc(cin, cin, cin, cin, t.data_ptr(), d2, 64, cout, cout, None) == \
        ssdc.SSDC_ERR_UNSUPPORTED
