"""ssd_complex_final_state: the state a scan leaves, without its rows of y.

Against the oracle's final state (the sequential scan in complex128) at each
precision's tolerance (relative Frobenius error: 1e-5 exact fp32, 2e-3 TF32),
on every chunk size, N and D below 64, ragged tails, T < Q, T = 1, a real x,
an initial state (also passed as the output buffer itself, in place), and
more sequences than SMs. The TF32 path runs the tensor-memory forward kernel's
state side alone, and the exact and staged paths the forward's first two
launches, so each must equal the final state of the forward pass on the same
arguments bit for bit."""
import numpy as np
import pytest
import torch

from oracle import naive_scan, naive_scan_inputs
from state_space_sequence_complex_gb300 import inputs, ssdc
from tests.gpu_util import assert_close, to_device

pytestmark = pytest.mark.gpu

STATE_ORDER = ["x_re", "x_im", "A_re", "A_im", "B_re", "B_im", "dt"]
FWD_ORDER = ["x_re", "x_im", "A_re", "A_im", "B_re", "B_im", "C_re", "C_im", "dt"]


@pytest.fixture(scope="module", autouse=True)
def built():
    from state_space_sequence_complex_gb300 import build
    build.build()
    ssdc.load()


def cplx(re, im):
    return re.double().cpu().numpy() + 1j * im.double().cpu().numpy()


def run_state(t, dims, Q, precision, s0=None, in_place=False):
    f = ssdc.FinalState(*dims, Q, precision)
    kw = {}
    if s0 is not None:
        if in_place:
            f.fs_re.copy_(s0[0])
            f.fs_im.copy_(s0[1])
            kw = dict(s0_re=f.fs_re, s0_im=f.fs_im)
        else:
            kw = dict(s0_re=s0[0], s0_im=s0[1])
    fs_re, fs_im = f(*[t[k] for k in STATE_ORDER], **kw)
    torch.cuda.synchronize()
    st = f.status()
    assert st == ssdc.SSDC_OK, ssdc.strerror(st)
    return cplx(fs_re, fs_im)


def state0(inp, seed):
    Bn, T, H, N, D = inp.dims
    rng = np.random.default_rng(seed)
    s0 = 8.0 * np.sqrt(0.5) * (rng.standard_normal((Bn, H, N, D)) + 1j * rng.standard_normal((Bn, H, N, D)))
    s0 = s0.real.astype(np.float32) + 1j * s0.imag.astype(np.float32)
    dev = (torch.from_numpy(np.ascontiguousarray(s0.real)).cuda(), torch.from_numpy(np.ascontiguousarray(s0.imag)).cuda())
    return s0.astype(np.complex128), dev


# (precision, B, T, H, D, N, Q)
CASES = [
    ("tf32", 2, 2048, 16, 64, 64, 64),
    ("tf32", 2, 300, 3, 64, 64, 16),
    ("tf32", 2, 333, 4, 40, 16, 32),
    ("tf32", 2, 64 * 9 + 13, 3, 64, 64, 128),
    ("tf32", 2, 511, 3, 24, 56, 256),
    ("tf32", 20, 200, 8, 64, 64, 64),   # 160 sequences: CTAs that walk two
    ("tf32", 1, 10, 2, 64, 64, 64),     # T < Q
    ("tf32", 1, 1, 2, 8, 8, 16),        # T = 1
    ("fp32", 2, 300, 3, 64, 64, 64),
    ("fp32", 1, 128, 2, 8, 8, 16),
    ("fp32", 2, 333, 3, 24, 40, 128),
    ("tf32_staged", 2, 300, 3, 64, 64, 64),
    ("tf32_staged", 2, 300, 3, 64, 64, 256),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "{}-B{}T{}H{}D{}N{}Q{}".format(*c))
def test_final_state_matches_oracle(case):
    precision, Bn, T, H, D, N, Q = case
    inp = inputs.custom(Bn, T, H, D, N, seed=9500 + T + Q)
    _, s_ref = naive_scan_inputs(inp)
    s = run_state(to_device(inp), inp.dims, Q, precision)
    expect = "state_tmem" if precision == "tf32" else ("staged_fp32" if precision == "fp32" else "staged_tf32")
    assert ssdc.last_path() == expect
    assert ssdc.last_launch_count() == (1 if precision == "tf32" else 2)
    assert_close(s, s, s_ref, s_ref, precision, f"final state alone {case}")


@pytest.mark.parametrize("precision,Q", [("tf32", 64), ("tf32", 128), ("fp32", 64)])
def test_initial_state_and_in_place(precision, Q):
    inp = inputs.custom(3, 330, 5, 64, 64, seed=9600 + Q)
    s0, s0_dev = state0(inp, 9601)
    _, s_ref = naive_scan_inputs(inp, s0=s0)
    t = to_device(inp)
    for in_place in (False, True):
        s = run_state(t, inp.dims, Q, precision, s0=s0_dev, in_place=in_place)
        assert_close(s, s, s_ref, s_ref, precision, f"final state alone from an initial state, in place {in_place}")


def test_real_x():
    inp = inputs.custom(2, 300, 4, 64, 64, seed=9700)
    _, s_ref = naive_scan(inp.x_re, np.zeros_like(inp.x_re), inp.A_re, inp.A_im, inp.B_re, inp.B_im, inp.C_re,
                          inp.C_im, inp.dt)
    t = to_device(inp)
    t["x_im"] = None
    s = run_state(t, inp.dims, 64, "tf32")
    assert_close(s, s, s_ref, s_ref, "tf32", "final state alone, real x")


@pytest.mark.parametrize("precision,Q,kernel", [("tf32", 64, 2), ("tf32", 16, 2), ("tf32", 256, 2),
                                                ("fp32", 64, 0), ("tf32_staged", 128, 0)])
def test_equals_the_forward_final_state(lib_option, precision, Q, kernel):
    """The same chunk states and state pass as the forward pass: its final state, bit for bit
    (the TF32 path against the tensor-memory kernel, forced)."""
    if kernel:
        lib_option(ssdc.OPT_FUSED_KERNEL, kernel)
    inp = inputs.custom(6, 700, 16, 64, 64, seed=9800 + Q)
    t = to_device(inp)
    s0, s0_dev = state0(inp, 9801)
    f = ssdc.Forward(*inp.dims, Q, precision)
    _, _, fs_re, fs_im = f(*[t[k] for k in FWD_ORDER], s0_re=s0_dev[0], s0_im=s0_dev[1])
    torch.cuda.synchronize()
    assert f.status() == ssdc.SSDC_OK
    if kernel:
        assert ssdc.last_path() == "fused_tmem"
    s_fwd = cplx(fs_re, fs_im)
    s = run_state(t, inp.dims, Q, precision, s0=s0_dev)
    assert np.array_equal(s, s_fwd)
