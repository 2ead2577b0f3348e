"""Real x (NEXT-2, the real-input half): x.im = NULL, as in the model, where x is
a real H*D slice of the input projection. The library then reads only x.re.
Checked against the oracle's scan with a zero imaginary plane, on every path
(exact fp32, staged TF32, the fused kernel at each cluster size, the host-buffer
and initial-state entry points), and for bit-identity with the same call given
an explicit zero plane."""
import numpy as np
import pytest
import torch

from oracle import naive_scan
from state_space_sequence_complex_gb300 import inputs, ssdc
from tests.gpu_util import assert_close, to_device

pytestmark = pytest.mark.gpu

ORDER = ["x_re", "x_im", "A_re", "A_im", "B_re", "B_im", "C_re", "C_im", "dt"]


@pytest.fixture(scope="module", autouse=True)
def built():
    from state_space_sequence_complex_gb300 import build
    build.build()
    ssdc.load()


def oracle_real(inp):
    return naive_scan(inp.x_re, np.zeros_like(inp.x_re), inp.A_re, inp.A_im, inp.B_re, inp.B_im,
                      inp.C_re, inp.C_im, inp.dt)


def run(inp, Q, precision, x_im="none"):
    t = to_device(inp)
    args = [t[k] for k in ORDER]
    args[1] = None if x_im == "none" else torch.zeros_like(t["x_re"])
    f = ssdc.Forward(*inp.dims, Q, precision)
    y_re, y_im, fs_re, fs_im = f(*args)
    torch.cuda.synchronize()
    st = f.status()
    assert st == ssdc.SSDC_OK, ssdc.strerror(st)
    y = y_re.double().cpu().numpy() + 1j * y_im.double().cpu().numpy()
    s = fs_re.double().cpu().numpy() + 1j * fs_im.double().cpu().numpy()
    return y, s


CASES = [
    (1, 200, 2, 16, 16, 32, "fp32", 0),
    (2, 300, 2, 64, 64, 64, "tf32_staged", 0),
    (1, 200, 2, 64, 64, 128, "tf32", 0),
    (2, 320, 3, 64, 64, 64, "tf32", 1),
    (2, 330, 3, 64, 64, 64, "tf32", 2),
    (2, 640, 3, 64, 64, 64, "tf32", 4),
    (1, 640, 2, 64, 64, 64, "tf32", 8),
    (1, 200, 2, 16, 16, 32, "tf32", 0),
    (2, 330, 3, 64, 64, 64, "tf32", -1),
    (20, 200, 8, 64, 64, 64, "tf32", -1),
    (20, 300, 8, 64, 64, 128, "tf32", -1),
    (2, 600, 3, 64, 64, 256, "tf32", -1),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}T{}H{}D{}N{}Q{}-{}-CL{}".format(*c))
def test_real_x_matches_oracle_and_zero_plane(case, lib_option):
    Bn, T, H, D, N, Q, precision, cl = case
    if cl > 0:
        lib_option(ssdc.OPT_FUSED_CLUSTER, cl)
    elif cl < 0:  # the fused kernel with the state in tensor memory
        lib_option(ssdc.OPT_FUSED_KERNEL, 2)
    inp = inputs.custom(Bn, T, H, D, N, seed=500 + T + H)
    y_ref, s_ref = oracle_real(inp)
    y, s = run(inp, Q, precision)
    assert_close(y, s, y_ref, s_ref, "fp32" if precision == "fp32" else "tf32", "real x")
    yz, sz = run(inp, Q, precision, x_im="zeros")
    assert np.array_equal(y, yz) and np.array_equal(s, sz)


def test_real_x_host_buffers_and_initial_state():
    inp = inputs.custom(2, 768, 3, 64, 64, seed=561)
    y_ref, s_ref = oracle_real(inp)
    h = {k: torch.from_numpy(np.ascontiguousarray(v)).pin_memory() for k, v in inp.arrays().items()}
    f = ssdc.HostForward(*inp.dims, 64, "tf32")
    args = [h[k] for k in ORDER]
    args[1] = None
    y_re, y_im, fs_re, fs_im = f(*args)  # 4 segments carried by the initial-state path
    y = y_re.double().numpy() + 1j * y_im.double().numpy()
    s = fs_re.double().numpy() + 1j * fs_im.double().numpy()
    assert_close(y, s, y_ref, s_ref, "tf32", "real x, host buffers")
