"""Parity of the backward pass (ssd_complex_bwd, exact fp32) with the gradient
oracle: every input gradient, element by element, on seeded inputs and output
gradients. Cases span several chunks with a ragged tail, every chunk size,
N and D from 8 to 64, a single partial chunk, T = 1, an initial state, a zero
final-state gradient, a real x and a loss of Re(y) alone; then the
single-layer size, and the differentiable scan (ssd_complex_scan) seeded by
autograd with the true output gradients."""
import numpy as np
import pytest
import torch

from oracle import naive_grad_inputs
from state_space_sequence_complex_gb300 import inputs, ssdc
from tests.gpu_util import rel_fro, to_device

pytestmark = pytest.mark.gpu

ORDER = ["x_re", "x_im", "A_re", "A_im", "B_re", "B_im", "C_re", "C_im", "dt"]
# Bound for the exact fp32 path. dx, dB_t, dC_t and d_initial_state: relative Frobenius
# error (sums of at most Q + N + D fp32 products; a few 1e-7 in practice). ddt and dA
# derive from dz_t, a sum of per-token terms r_t = <dC_t, C_t> - <dB_t, B_t> that cancel:
# dz_t is exactly zero at T = 1, and the sum over tokens that gives dA cancels by factors
# of 10 to 500 on these inputs. Their error is therefore bounded relative to the size of
# the terms summed, m_t = |dz_t| + |<dC_t, C_t>| + |<dB_t, B_t>| (oracle values):
#   ||ddt - ddt_ref|| <= TOL_BWD * || |A| sigmoid(dt_t) m_t ||,
#   |dA_h - dA_ref_h| <= TOL_BWD * sum_{b,t} softplus(dt_t) m_t.
TOL_BWD = 1e-5


@pytest.fixture(scope="module", autouse=True)
def built():
    from state_space_sequence_complex_gb300 import build
    build.build()
    ssdc.load()


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def run_bwd(inp, og, Q, s0=None, with_dfs=True, real_x=False, dy_imag=True, backward=None):
    t = to_device(inp)
    if real_x:
        t["x_im"] = None
    b = backward or ssdc.Backward(*inp.dims, Q)
    kw = {}
    if s0 is not None:
        kw = dict(s0_re=cuda(s0.real), s0_im=cuda(s0.imag))
    g = b(*[t[k] for k in ORDER], cuda(og.dy_re), cuda(og.dy_im) if dy_imag else None,
          cuda(og.dfs_re) if with_dfs else None, cuda(og.dfs_im) if with_dfs else None, **kw)
    torch.cuda.synchronize()
    st = ssdc.ssd_complex_status(b.workspace)
    assert st == ssdc.SSDC_OK, ssdc.strerror(st)
    n = lambda k: g[k].double().cpu().numpy()
    out = {"dA": n("dA_re") + 1j * n("dA_im"), "dB": n("dB_re") + 1j * n("dB_im"),
           "dC": n("dC_re") + 1j * n("dC_im"), "ddt": n("ddt")}
    out["dx"] = n("dx_re") + (0 if real_x else 1j * n("dx_im"))
    if s0 is not None:
        out["ds0"] = n("ds0_re") + 1j * n("ds0_im")
    return out


def oracle_grads(inp, og, s0=None, with_dfs=True, real_x=False, dy_imag=True):
    if real_x:
        inp = inputs.Inputs(**dict(inp.arrays(), x_im=np.zeros_like(inp.x_im)))
    dy = og.dy_re.astype(np.float64) + (1j * og.dy_im if dy_imag else 0)
    dfs = og.dfs_re + 1j * og.dfs_im if with_dfs else None
    s0_32 = None
    if s0 is not None:  # the library reads the initial state in float32
        s0_32 = s0.real.astype(np.float32).astype(np.float64) + 1j * s0.imag.astype(np.float32)
    g = naive_grad_inputs(inp, dy, dfs, s0=s0_32)
    if real_x:
        g["dx"] = g["dx"].real
    return g


def term_scale(inp, ref):
    """m_t = |dz_t| + |<dC_t, C_t>| + |<dB_t, B_t>| (B,T,H) from the oracle's gradients."""
    c = inp.complex()
    dcc = np.abs((ref["dC"] * np.conj(c["C"])).sum(-1))
    dbb = np.abs((ref["dB"] * np.conj(c["B"])).sum(-1))
    return np.abs(ref["dz"]) + dcc + dbb


def check(got, ref, inp, what):
    """Errors of every gradient (relative, or relative to the term scale for ddt and
    dA); asserts each is within TOL_BWD."""
    errs = {}
    for k, v in got.items():
        assert np.all(np.isfinite(v)), f"{what}: non-finite {k}"
        if k not in ("ddt", "dA"):
            errs[k] = rel_fro(v, ref[k])
    m = term_scale(inp, ref)
    dt = inp.dt.astype(np.float64)
    A = np.abs(inp.complex()["A"])
    if "ddt" in got:
        scale = np.linalg.norm((A * m / (1.0 + np.exp(-dt))).ravel())
        errs["ddt"] = float(np.linalg.norm((got["ddt"] - ref["ddt"]).ravel()) / scale)
    if "dA" in got:
        scale = (np.logaddexp(0.0, dt) * m).sum(axis=(0, 1))
        errs["dA"] = float(np.max(np.abs(got["dA"] - ref["dA"]) / scale))
    bad = {k: e for k, e in errs.items() if e > TOL_BWD}
    assert not bad, f"{what}: errors {errs}"
    return errs


def state(inp, seed):
    Bn, T, H, N, D = inp.dims
    r, i = inputs.initial_state(Bn, H, N, D, seed)
    return 8.0 * (r.astype(np.float64) + 1j * i)  # of the size of a state after a few dozen tokens


# (B, T, H, D, N, Q): ragged tails at every chunk size, T < Q, T = 1
CASES = [
    (1, 200, 2, 16, 16, 32),
    (2, 130, 3, 8, 24, 16),
    (1, 256, 2, 64, 64, 64),
    (2, 320, 2, 64, 64, 128),
    (1, 600, 2, 32, 64, 256),
    (3, 100, 2, 64, 8, 64),
    (1, 40, 2, 16, 16, 64),
    (2, 1, 2, 8, 8, 16),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}T{}H{}D{}N{}Q{}".format(*c))
def test_backward_matches_oracle(case):
    Bn, T, H, D, N, Q = case
    inp = inputs.custom(Bn, T, H, D, N, seed=500 + T + N)
    og = inputs.output_grads(Bn, T, H, D, N, seed=600 + T)
    check(run_bwd(inp, og, Q), oracle_grads(inp, og), inp, f"case {case}")


@pytest.mark.parametrize("case", [(2, 200, 2, 16, 16, 64), (1, 300, 2, 64, 64, 128)],
                         ids=["Q64", "Q128"])
def test_backward_with_initial_state(case):
    Bn, T, H, D, N, Q = case
    inp = inputs.custom(Bn, T, H, D, N, seed=700 + T)
    og = inputs.output_grads(Bn, T, H, D, N, seed=701)
    s0 = state(inp, 702)
    check(run_bwd(inp, og, Q, s0=s0), oracle_grads(inp, og, s0=s0), inp, f"initial state {case}")


def test_backward_real_x_and_real_loss():
    """x real (x.im null: dx.re only) and a loss of Re(y) alone (dy.im null) with no
    final-state gradient: the model's case."""
    Bn, T, H, D, N, Q = 2, 190, 3, 32, 16, 64
    inp = inputs.custom(Bn, T, H, D, N, seed=800)
    og = inputs.output_grads(Bn, T, H, D, N, seed=801)
    kw = dict(with_dfs=False, real_x=True, dy_imag=False)
    check(run_bwd(inp, og, Q, **kw), oracle_grads(inp, og, **kw), inp, "real x, Re(y) loss")


def test_backward_zero_output_grads_give_zero():
    Bn, T, H, D, N, Q = 1, 150, 2, 16, 16, 32
    inp = inputs.custom(Bn, T, H, D, N, seed=810)
    og = inputs.output_grads(Bn, T, H, D, N, seed=811)
    zero = inputs.OutputGrads(*[np.zeros_like(a) for a in (og.dy_re, og.dy_im, og.dfs_re, og.dfs_im)])
    g = run_bwd(inp, zero, Q)
    for k, v in g.items():
        assert np.all(v == 0.0), k


def test_backward_repeated_calls_are_bitwise_identical():
    inp = inputs.custom(2, 333, 2, 64, 64, seed=820)
    og = inputs.output_grads(2, 333, 2, 64, 64, seed=821)
    b = ssdc.Backward(*inp.dims, 64)
    g1 = run_bwd(inp, og, 64, backward=b)
    g2 = run_bwd(inp, og, 64, backward=b)
    for k in g1:
        assert np.array_equal(g1[k], g2[k]), k
    assert ssdc.last_launch_count() == 5


def test_backward_single_layer_matches_oracle():
    inp = inputs.generate(inputs.LAYER)
    Bn, T, H, N, D = inp.dims
    og = inputs.output_grads(Bn, T, H, D, N, seed=830)
    errs = check(run_bwd(inp, og, 64), oracle_grads(inp, og), inp, "single layer")
    assert max(errs.values()) <= TOL_BWD


def test_scan_autograd_matches_oracle():
    """ssd_complex_scan under autograd, with a loss whose output gradients are random
    (not all ones) and with an initial state: every input gets its gradient."""
    Bn, T, H, D, N, Q = 2, 170, 2, 16, 32, 32
    inp = inputs.custom(Bn, T, H, D, N, seed=840)
    og = inputs.output_grads(Bn, T, H, D, N, seed=841)
    s0 = state(inp, 842)
    leaves = {k: cuda(v).requires_grad_(True) for k, v in inp.arrays().items()}
    s0_re, s0_im = cuda(s0.real).requires_grad_(True), cuda(s0.imag).requires_grad_(True)
    y_re, y_im, fs_re, fs_im = ssdc.ssd_complex_scan(*[leaves[k] for k in ORDER], Q,
                                                     s0_re=s0_re, s0_im=s0_im, precision="fp32")
    loss = ((y_re * cuda(og.dy_re)).sum() + (y_im * cuda(og.dy_im)).sum()
            + (fs_re * cuda(og.dfs_re)).sum() + (fs_im * cuda(og.dfs_im)).sum())
    loss.backward()
    for k, v in list(leaves.items()) + [("s0_re", s0_re), ("s0_im", s0_im)]:
        assert v.grad is not None, f"no gradient for {k}"
        assert torch.isfinite(v.grad).all(), k
        assert v.grad.abs().sum() > 0, f"zero gradient for {k}"
    ref = oracle_grads(inp, og, s0=s0)
    n = lambda t: t.grad.double().cpu().numpy()
    got = {"dx": n(leaves["x_re"]) + 1j * n(leaves["x_im"]),
           "dA": n(leaves["A_re"]) + 1j * n(leaves["A_im"]),
           "dB": n(leaves["B_re"]) + 1j * n(leaves["B_im"]),
           "dC": n(leaves["C_re"]) + 1j * n(leaves["C_im"]),
           "ddt": n(leaves["dt"]), "ds0": n(s0_re) + 1j * n(s0_im)}
    check(got, ref, inp, "autograd")


def test_scan_autograd_real_x_loss_of_re_y():
    """The model's use: x real, the loss reads Re(y) only (autograd hands the function
    zero gradients for y.im and the final state)."""
    Bn, T, H, D, N, Q = 1, 128, 2, 64, 64, 64
    inp = inputs.custom(Bn, T, H, D, N, seed=850)
    og = inputs.output_grads(Bn, T, H, D, N, seed=851)
    arrs = inp.arrays()
    leaves = {k: cuda(v).requires_grad_(True) for k, v in arrs.items() if k != "x_im"}
    y_re, _, _, _ = ssdc.ssd_complex_scan(leaves["x_re"], None, leaves["A_re"], leaves["A_im"],
                                          leaves["B_re"], leaves["B_im"], leaves["C_re"],
                                          leaves["C_im"], leaves["dt"], Q, precision="tf32")
    (y_re * cuda(og.dy_re)).sum().backward()
    ref = oracle_grads(inp, og, with_dfs=False, real_x=True, dy_imag=False)
    n = lambda t: t.grad.double().cpu().numpy()
    got = {"dx": n(leaves["x_re"]), "dA": n(leaves["A_re"]) + 1j * n(leaves["A_im"]),
           "dB": n(leaves["B_re"]) + 1j * n(leaves["B_im"]),
           "dC": n(leaves["C_re"]) + 1j * n(leaves["C_im"]), "ddt": n(leaves["dt"])}
    check(got, ref, inp, "autograd, real x")


@pytest.mark.parametrize("Q", [64, 256])
def test_backward_long_sequence(Q):
    """The long-memory workload's length (T = 65536: 1024 chunks at Q = 64) with its
    slow decays, at N = D = 8 so that the oracle's stored states stay small: both chunk
    recurrences run the full length, and dz is anchored in every chunk."""
    Bn, T, H, D, N = 1, 65536, 2, 8, 8
    inp = inputs.custom(Bn, T, H, D, N, seed=860 + Q, dt_mean=-2.0, dt_std=0.5,
                        re_lo=-0.1, re_hi=-0.01)
    og = inputs.output_grads(Bn, T, H, D, N, seed=861)
    s0 = state(inp, 862)
    check(run_bwd(inp, og, Q, s0=s0), oracle_grads(inp, og, s0=s0), inp, f"long sequence Q{Q}")


def test_backward_dt_zero_and_growing_states():
    """dt = 0 everywhere (A_bar = 2^A at every token) and Re(A) > 0 (the pages' Skill-2
    example draws Re(A) around -1 with a tail above zero: the states grow), the latter on
    a short sequence, where growth stays within fp32 range."""
    Bn, T, H, D, N, Q = 2, 200, 2, 16, 16, 32
    inp = inputs.custom(Bn, T, H, D, N, seed=870, dt_mode="zero")
    og = inputs.output_grads(Bn, T, H, D, N, seed=871)
    check(run_bwd(inp, og, Q), oracle_grads(inp, og), inp, "dt = 0")
    Bn, T = 1, 48
    inp = inputs.custom(Bn, T, H, D, N, seed=872, re_lo=0.01, re_hi=0.1)
    og = inputs.output_grads(Bn, T, H, D, N, seed=873)
    check(run_bwd(inp, og, 16), oracle_grads(inp, og), inp, "Re(A) > 0")


def test_scan_autograd_through_segments():
    """Two segments chained through the carried state (the second starts from the first's
    final state), A shared between them: autograd through both calls gives the whole
    sequence's gradients; dA accumulates over the two calls."""
    Bn, T, H, D, N, Q, T1 = 1, 256, 2, 16, 16, 32, 128
    inp = inputs.custom(Bn, T, H, D, N, seed=880)
    og = inputs.output_grads(Bn, T, H, D, N, seed=881)
    arrs = inp.arrays()
    A_re = cuda(arrs["A_re"]).requires_grad_(True)
    A_im = cuda(arrs["A_im"]).requires_grad_(True)
    seg = lambda a, b: {k: cuda(v[:, a:b]).requires_grad_(True) for k, v in arrs.items() if v.ndim > 1}
    s1, s2 = seg(0, T1), seg(T1, T)
    args = lambda s: (s["x_re"], s["x_im"], A_re, A_im, s["B_re"], s["B_im"], s["C_re"], s["C_im"], s["dt"])
    y1r, y1i, f1r, f1i = ssdc.ssd_complex_scan(*args(s1), Q, precision="fp32")
    y2r, y2i, f2r, f2i = ssdc.ssd_complex_scan(*args(s2), Q, s0_re=f1r, s0_im=f1i, precision="fp32")
    gy_re, gy_im = cuda(og.dy_re), cuda(og.dy_im)
    loss = ((y1r * gy_re[:, :T1]).sum() + (y1i * gy_im[:, :T1]).sum() + (y2r * gy_re[:, T1:]).sum()
            + (y2i * gy_im[:, T1:]).sum() + (f2r * cuda(og.dfs_re)).sum() + (f2i * cuda(og.dfs_im)).sum())
    loss.backward()
    ref = oracle_grads(inp, og)
    n = lambda t: t.grad.double().cpu().numpy()
    cat = lambda k: np.concatenate([n(s1[k]), n(s2[k])], axis=1)
    got = {"dx": cat("x_re") + 1j * cat("x_im"), "dB": cat("B_re") + 1j * cat("B_im"),
           "dC": cat("C_re") + 1j * cat("C_im"), "ddt": cat("dt"), "dA": n(A_re) + 1j * n(A_im)}
    check(got, ref, inp, "autograd through two segments")


def test_scan_autograd_staged_forward():
    """The staged TF32 forward (Q = 128) under autograd: the exact backward does not depend
    on the forward's precision."""
    Bn, T, H, D, N, Q = 1, 300, 2, 64, 64, 128
    inp = inputs.custom(Bn, T, H, D, N, seed=890)
    og = inputs.output_grads(Bn, T, H, D, N, seed=891)
    leaves = {k: cuda(v).requires_grad_(True) for k, v in inp.arrays().items()}
    y_re, y_im, fs_re, fs_im = ssdc.ssd_complex_scan(*[leaves[k] for k in ORDER], Q, precision="tf32")
    loss = ((y_re * cuda(og.dy_re)).sum() + (y_im * cuda(og.dy_im)).sum()
            + (fs_re * cuda(og.dfs_re)).sum() + (fs_im * cuda(og.dfs_im)).sum())
    loss.backward()
    ref = oracle_grads(inp, og)
    n = lambda t: t.grad.double().cpu().numpy()
    got = {"dx": n(leaves["x_re"]) + 1j * n(leaves["x_im"]),
           "dA": n(leaves["A_re"]) + 1j * n(leaves["A_im"]),
           "dB": n(leaves["B_re"]) + 1j * n(leaves["B_im"]),
           "dC": n(leaves["C_re"]) + 1j * n(leaves["C_im"]), "ddt": n(leaves["dt"])}
    check(got, ref, inp, "autograd, staged TF32 forward")
