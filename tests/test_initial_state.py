"""The forward pass from a given initial state (ssd_complex_fwd_init): the
scan with s_{-1} = S0 instead of zero, so that a sequence can be processed in
segments. Checked against the oracle's scan from the same initial state (the
oracle's initial-state path is itself pinned by the continuation invariant on
the CPU), on every path: exact fp32, staged TF32 and the fused TF32 kernel at
each cluster size, including clusters that own several sequences. Then
segment continuation through the library: [0, T1) and then [T1, T) from the
carried state, in place, against the whole scan."""
import numpy as np
import pytest
import torch

from oracle import naive_scan_inputs
from state_space_sequence_complex_gb300 import inputs, ssdc
from tests.gpu_util import TOL, assert_close, rel_fro, to_device

pytestmark = pytest.mark.gpu

ORDER = ["x_re", "x_im", "A_re", "A_im", "B_re", "B_im", "C_re", "C_im", "dt"]


@pytest.fixture(scope="module", autouse=True)
def built():
    from state_space_sequence_complex_gb300 import build
    build.build()
    ssdc.load()


def random_state(inp, seed):
    Bn, T, H, N, D = inp.dims
    rng = np.random.default_rng(seed)
    s = np.sqrt(0.5) * 8.0  # of the size of a state after a few dozen tokens
    return (rng.standard_normal((Bn, H, N, D)) * s + 1j * rng.standard_normal((Bn, H, N, D)) * s)


def run(inp, Q, precision, s0=None, forward=None):
    t = to_device(inp)
    f = forward or ssdc.Forward(*inp.dims, Q, precision)
    kw = {}
    if s0 is not None:
        kw = dict(s0_re=torch.from_numpy(np.ascontiguousarray(s0.real, dtype=np.float32)).cuda(),
                  s0_im=torch.from_numpy(np.ascontiguousarray(s0.imag, dtype=np.float32)).cuda())
    y_re, y_im, fs_re, fs_im = f(*[t[k] for k in ORDER], **kw)
    torch.cuda.synchronize()
    st = f.status()
    assert st == ssdc.SSDC_OK, ssdc.strerror(st)
    y = y_re.double().cpu().numpy() + 1j * y_im.double().cpu().numpy()
    s = fs_re.double().cpu().numpy() + 1j * fs_im.double().cpu().numpy()
    return y, s


def oracle(inp, s0):
    # the oracle takes the initial state at the precision the library reads it in
    s0_32 = s0.real.astype(np.float32).astype(np.float64) + 1j * s0.imag.astype(np.float32).astype(np.float64)
    return naive_scan_inputs(inp, s0=s0_32)


# (B, T, H, D, N, Q, precision, cluster; -1: the tensor-memory kernel): T not a multiple of Q in several; 40 sequences
# at clusters of 4 and 8 give clusters that own two sequences (a state from the last CTA
# of the cluster follows an initial state in the first CTA's buffer).
CASES = [
    (1, 200, 2, 16, 16, 32, "fp32", 0),
    (2, 130, 3, 8, 24, 16, "fp32", 0),
    (2, 300, 2, 64, 64, 64, "tf32_staged", 0),
    (1, 200, 2, 64, 64, 128, "tf32", 0),
    (2, 320, 3, 64, 64, 64, "tf32", 1),
    (2, 330, 3, 64, 64, 64, "tf32", 2),
    (2, 640, 3, 64, 64, 64, "tf32", 4),
    (1, 640, 2, 64, 64, 64, "tf32", 8),
    (5, 640, 8, 64, 64, 64, "tf32", 4),
    (5, 640, 8, 64, 64, 64, "tf32", 8),
    (5, 136, 8, 64, 64, 64, "tf32", 4),
    (1, 200, 2, 16, 16, 32, "tf32", 0),
    (2, 130, 3, 8, 24, 16, "tf32", 0),
    (2, 330, 3, 64, 64, 64, "tf32", -1),
    (20, 200, 8, 64, 64, 64, "tf32", -1),
    (20, 136, 8, 64, 64, 32, "tf32", -1),
    (20, 300, 8, 64, 64, 128, "tf32", -1),
    (2, 600, 3, 64, 64, 256, "tf32", -1),
    (2, 130, 3, 8, 24, 128, "tf32", -1),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}T{}H{}D{}N{}Q{}-{}-CL{}".format(*c))
def test_initial_state_matches_oracle(case, lib_option):
    Bn, T, H, D, N, Q, precision, cl = case
    if cl > 0:
        lib_option(ssdc.OPT_FUSED_CLUSTER, cl)
    elif cl < 0:  # the fused kernel with the state in tensor memory
        lib_option(ssdc.OPT_FUSED_KERNEL, 2)
    inp = inputs.custom(Bn, T, H, D, N, seed=400 + T + H)
    s0 = random_state(inp, seed=T)
    y_ref, s_ref = oracle(inp, s0)
    y, s = run(inp, Q, precision, s0=s0)
    assert_close(y, s, y_ref, s_ref, "fp32" if precision == "fp32" else "tf32", "initial state")


@pytest.mark.parametrize("precision", ["fp32", "tf32"])
def test_zero_initial_state_is_the_plain_scan(precision):
    inp = inputs.custom(2, 256, 3, 64, 64, seed=431)
    y0, s0 = run(inp, 64, precision)
    y1, s1 = run(inp, 64, precision, s0=np.zeros((2, 3, 64, 64), complex))
    assert np.array_equal(y0, y1) and np.array_equal(s0, s1)


@pytest.mark.parametrize("precision,cl", [("fp32", 0), ("tf32", 1), ("tf32", 4), ("tf32", -1)])
def test_segments_continue_in_place(precision, cl, lib_option):
    """[0, T1) then [T1, T) started from the carried final state (the Forward's own
    final-state tensors passed back as the initial state) equals the whole scan."""
    if cl > 0:
        lib_option(ssdc.OPT_FUSED_CLUSTER, cl)
    elif cl < 0:  # the fused kernel with the state in tensor memory
        lib_option(ssdc.OPT_FUSED_KERNEL, 2)
    Bn, T, H, D, N, Q = 2, 768, 3, 64, 64, 64
    T1 = 320
    inp = inputs.custom(Bn, T, H, D, N, seed=441)
    y_ref, s_ref = naive_scan_inputs(inp)
    t = to_device(inp)
    seg = lambda a, b: [t[k] if t[k].dim() == 1 else t[k][:, a:b].contiguous() for k in ORDER]
    f1 = ssdc.Forward(Bn, T1, H, N, D, Q, precision)
    f2 = ssdc.Forward(Bn, T - T1, H, N, D, Q, precision)
    y1 = f1(*seg(0, T1))
    ya = (y1[0].double() + 1j * y1[1].double()).cpu().numpy()
    f2.fs_re.copy_(f1.fs_re)
    f2.fs_im.copy_(f1.fs_im)
    y2 = f2(*seg(T1, T), s0_re=f2.fs_re, s0_im=f2.fs_im)  # in place
    torch.cuda.synchronize()
    assert f1.status() == ssdc.SSDC_OK and f2.status() == ssdc.SSDC_OK
    yb = (y2[0].double() + 1j * y2[1].double()).cpu().numpy()
    s = (f2.fs_re.double() + 1j * f2.fs_im.double()).cpu().numpy()
    assert_close(np.concatenate([ya, yb], axis=1), s, y_ref, s_ref, "fp32" if precision == "fp32" else "tf32",
                 "segments")
