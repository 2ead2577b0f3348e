"""Parity of the TF32 backward pass (ssd_complex_bwd with SSDC_PREC_TF32: the
per-chunk gradient products on the tensor cores) with the gradient oracle.
The bar is the TF32 forward's, 2e-3: relative Frobenius error for dx, dB_t,
dC_t and d_initial_state, and, for ddt and dA, error relative to the size of
the per-token terms their sums cancel (the scales of the exact backward's
tests). Cases: the single-layer size, every chunk size (128 and 256 worked
as 64-token chunks), N and D below 64, ragged tails, T = 1, an initial
state, no final-state gradient, a real x with a loss of Re(y) alone; and,
for the chunk kernel, which walks several chunks a CTA, Q below 64 and the
real x and loss with more chunks than SMs."""
import numpy as np
import pytest

from state_space_sequence_complex_gb300 import inputs, ssdc
from tests.gpu_util import RECORDED, rel_fro
from tests.test_backward_gpu import oracle_grads, run_bwd, state, term_scale

pytestmark = pytest.mark.gpu

TOL_TF32 = 2e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    from state_space_sequence_complex_gb300 import build
    build.build()
    ssdc.load()


def check_tf32(got, ref, inp, what):
    errs = {}
    for k, v in got.items():
        assert np.all(np.isfinite(v)), f"{what}: non-finite {k}"
        if k not in ("ddt", "dA"):
            errs[k] = rel_fro(v, ref[k])
    m = term_scale(inp, ref)
    dt = inp.dt.astype(np.float64)
    A = np.abs(inp.complex()["A"])
    scale = np.linalg.norm((A * m / (1.0 + np.exp(-dt))).ravel())
    errs["ddt"] = float(np.linalg.norm((got["ddt"] - ref["ddt"]).ravel()) / scale)
    scale = (np.logaddexp(0.0, dt) * m).sum(axis=(0, 1))
    errs["dA"] = float(np.max(np.abs(got["dA"] - ref["dA"]) / scale))
    RECORDED.append((what, "tf32 bwd", ", ".join(f"{k} {e:.1e}" for k, e in sorted(errs.items())),
                     max(errs.get("dx", 0), errs.get("dB", 0), errs.get("dC", 0)),
                     max(errs["ddt"], errs["dA"])))
    bad = {k: e for k, e in errs.items() if e > TOL_TF32}
    assert not bad, f"{what}: errors {errs}"
    return errs


def run_tf32(inp, og, Q, **kw):
    b = ssdc.Backward(*inp.dims, Q, precision="tf32")
    return run_bwd(inp, og, Q, backward=b, **kw)


# (B, T, H, D, N, Q)
CASES = [
    (2, 2048, 16, 64, 64, 64),
    (2, 200, 3, 64, 64, 64),
    (2, 257, 3, 64, 64, 32),
    (1, 130, 2, 8, 8, 16),
    (2, 333, 3, 40, 16, 64),
    (1, 1, 2, 64, 64, 64),
    (3, 100, 2, 24, 56, 32),
    (4, 1000, 16, 64, 64, 32),  # many chunks a CTA: the unloaded rows past Q zeroed again each chunk
    (3, 700, 16, 40, 24, 16),
    (1, 640, 16, 64, 64, 64),   # 160 chunks: 8 CTAs take two, the rest one
    (2, 300, 3, 64, 64, 128),   # Q = 128 and 256: worked as 64-token chunks
    (1, 600, 2, 32, 48, 256),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}T{}H{}D{}N{}Q{}".format(*c))
def test_tf32_backward_matches_gradient_oracle(case):
    Bn, T, H, D, N, Q = case
    inp = inputs.custom(Bn, T, H, D, N, seed=8000 + T + Q)
    og = inputs.output_grads(Bn, T, H, D, N, seed=8100 + T)
    got = run_tf32(inp, og, Q)
    check_tf32(got, oracle_grads(inp, og), inp, f"tf32 backward {case}")


def test_tf32_backward_initial_state_no_final_gradient():
    inp = inputs.custom(2, 300, 3, 64, 64, seed=8200)
    og = inputs.output_grads(2, 300, 3, 64, 64, seed=8201)
    s0 = state(inp, 8202)
    got = run_tf32(inp, og, 64, s0=s0, with_dfs=False)
    check_tf32(got, oracle_grads(inp, og, s0=s0, with_dfs=False), inp, "tf32 backward, initial state")


@pytest.mark.parametrize("Bn,T,H,Q", [(2, 256, 4, 64), (4, 1000, 16, 64), (4, 1000, 16, 32)])
def test_tf32_backward_real_x_and_real_loss(Bn, T, H, Q):
    # (4, 1000, 16): 1024 and 2048 chunks, several a CTA, so the imaginary planes (and at Q = 32 the
    # rows past Q) are zeroed again each chunk
    inp = inputs.custom(Bn, T, H, 64, 64, seed=8300 + T + Q)
    og = inputs.output_grads(Bn, T, H, 64, 64, seed=8301 + T + Q)
    got = run_tf32(inp, og, Q, real_x=True, dy_imag=False, with_dfs=False)
    ref = oracle_grads(inp, og, real_x=True, dy_imag=False, with_dfs=False)
    check_tf32(got, ref, inp, "tf32 backward, real x, Re(y) loss")


def test_tf32_backward_agrees_with_exact_backward():
    # the same call at both precisions: within the TF32 bar of each other, and bit-identical
    # when repeated
    inp = inputs.custom(2, 640, 8, 64, 64, seed=8400)
    og = inputs.output_grads(2, 640, 8, 64, 64, seed=8401)
    g32 = run_bwd(inp, og, 64)
    gtf = run_tf32(inp, og, 64)
    gtf2 = run_tf32(inp, og, 64)
    for k in ("dx", "dB", "dC"):
        assert rel_fro(gtf[k], g32[k]) <= TOL_TF32
        assert np.array_equal(gtf[k], gtf2[k])


def test_scan_autograd_with_tf32_backward():
    """ssd_complex_scan with the TF32 forward and the TF32 backward under autograd: a
    loss with random output gradients and an initial state; every input gets its
    gradient, within the TF32 bar of the gradient oracle."""
    from tests.test_backward_gpu import ORDER, cuda
    Bn, T, H, D, N, Q = 2, 170, 2, 16, 32, 32
    inp = inputs.custom(Bn, T, H, D, N, seed=8500)
    og = inputs.output_grads(Bn, T, H, D, N, seed=8501)
    s0 = state(inp, 8502)
    leaves = {k: cuda(v).requires_grad_(True) for k, v in inp.arrays().items()}
    s0_re, s0_im = cuda(s0.real).requires_grad_(True), cuda(s0.imag).requires_grad_(True)
    y_re, y_im, fs_re, fs_im = ssdc.ssd_complex_scan(*[leaves[k] for k in ORDER], Q, s0_re=s0_re, s0_im=s0_im,
                                                     precision="tf32", bwd_precision="tf32")
    loss = ((y_re * cuda(og.dy_re)).sum() + (y_im * cuda(og.dy_im)).sum()
            + (fs_re * cuda(og.dfs_re)).sum() + (fs_im * cuda(og.dfs_im)).sum())
    loss.backward()
    n = lambda t: t.grad.double().cpu().numpy()
    got = {"dx": n(leaves["x_re"]) + 1j * n(leaves["x_im"]), "dA": n(leaves["A_re"]) + 1j * n(leaves["A_im"]),
           "dB": n(leaves["B_re"]) + 1j * n(leaves["B_im"]), "dC": n(leaves["C_re"]) + 1j * n(leaves["C_im"]),
           "ddt": n(leaves["dt"]), "ds0": n(s0_re) + 1j * n(s0_im)}
    check_tf32(got, oracle_grads(inp, og, s0=s0), inp, "tf32 backward through autograd")


@pytest.mark.parametrize("Q", [64, 128])
def test_tf32_backward_long_sequence(Q):
    """The long-memory workload's length (T = 65536: 1024 chunks of 64 tokens in one sequence,
    all walked by one CTA after another) with its slow decays, at N = D = 8 so that the oracle's
    stored states stay small, from an initial state."""
    from tests.test_backward_gpu import state
    Bn, T, H, D, N = 1, 65536, 2, 8, 8
    inp = inputs.custom(Bn, T, H, D, N, seed=8700 + Q, dt_mean=-2.0, dt_std=0.5, re_lo=-0.1, re_hi=-0.01)
    og = inputs.output_grads(Bn, T, H, D, N, seed=8701)
    s0 = state(inp, 8702)
    got = run_tf32(inp, og, Q, s0=s0)
    check_tf32(got, oracle_grads(inp, og, s0=s0), inp, f"tf32 backward, long sequence Q{Q}")


def test_tf32_backward_dt_zero_and_growing_states():
    """dt = 0 everywhere (A_bar = 2^A at every token; the TF32 kernels' decay tables then
    hold exact powers) and Re(A) > 0 on a short sequence, where the states grow."""
    Bn, T, H, D, N, Q = 2, 200, 2, 16, 16, 32
    inp = inputs.custom(Bn, T, H, D, N, seed=8800, dt_mode="zero")
    og = inputs.output_grads(Bn, T, H, D, N, seed=8801)
    check_tf32(run_tf32(inp, og, Q), oracle_grads(inp, og), inp, "tf32 backward, dt = 0")
    Bn, T = 1, 48
    inp = inputs.custom(Bn, T, H, D, N, seed=8802, re_lo=0.01, re_hi=0.1)
    og = inputs.output_grads(Bn, T, H, D, N, seed=8803)
    check_tf32(run_tf32(inp, og, 16), oracle_grads(inp, og), inp, "tf32 backward, Re(A) > 0")
