"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these expected values comes from the oracle itself: each is a
brute-force O(T^2) materialisation of the SSD matrix, a closed form, a library
routine (scipy's IIR filter), an invariant, the independent chunkwise form in
``chunkwise_ref`` or a value printed on the pages (``tests/golden``).
"""
import os

import numpy as np
import pytest
import scipy.signal

from oracle import naive_scan
from state_space_sequence_complex_gb300 import inputs
from tests.chunkwise_ref import chunkwise

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rel_fro(a, b):
    return np.linalg.norm((a - b).ravel()) / max(np.linalg.norm(np.ravel(b)), 1e-300)


def planes(c):
    c = np.asarray(c)
    return np.ascontiguousarray(c.real, np.float32), np.ascontiguousarray(c.imag, np.float32)


def run(x, A, Bt, Ct, dt, **kw):
    xr, xi = planes(x)
    ar, ai = planes(A)
    br, bi = planes(Bt)
    cr, ci = planes(Ct)
    return naive_scan(xr, xi, ar, ai, br, bi, cr, ci, np.asarray(dt, np.float32), **kw)


def f32c(c):
    """Round a complex array to complex64 and back, as the oracle reads it."""
    return np.asarray(c).astype(np.complex64).astype(np.complex128)


def rand_case(Bn=2, T=24, H=2, N=3, D=4, seed=7, dt_mode="normal"):
    inp = inputs.custom(Bn, T, H, D, N, seed, dt_mode=dt_mode)
    c = inp.complex()
    return c["x"], c["A"], c["B"], c["C"], c["dt"]


def brute_force(x, A, Bt, Ct, dt):
    """Materialised SSD matrix: y_t = sum_{s<=t} (C_t . B_s) prod_{k=s+1..t} Abar_k x_s."""
    Bn, T, H, D = x.shape
    delta = np.logaddexp(0.0, dt)                 # softplus, via a library routine
    abar = np.exp(delta * A[None, None, :])       # (B,T,H)
    y = np.zeros_like(x)
    st = np.zeros((Bn, H, Bt.shape[-1], D), complex)
    for b in range(Bn):
        for h in range(H):
            for t in range(T):
                for s in range(t + 1):
                    decay = np.prod(abar[b, s + 1:t + 1, h])
                    y[b, t, h] += np.dot(Ct[b, t, h], Bt[b, s, h]) * decay * x[b, s, h]
            for s in range(T):
                decay = np.prod(abar[b, s + 1:T, h])
                st[b, h] += decay * np.outer(Bt[b, s, h], x[b, s, h])
    return y, st


@pytest.mark.parametrize("dt_mode", ["normal", "zero"])
def test_matches_bruteforce_ssd_matrix(dt_mode):
    x, A, Bt, Ct, dt = rand_case(dt_mode=dt_mode)
    y, s = run(x, A, Bt, Ct, dt)
    yb, sb = brute_force(x, A, Bt, Ct, dt)
    assert rel_fro(y, yb) < 1e-12
    assert rel_fro(s, sb) < 1e-12


def test_single_step_closed_form():
    x, A, Bt, Ct, dt = rand_case(Bn=3, T=1, H=4, N=5, D=6)
    y, s = run(x, A, Bt, Ct, dt)
    # T = 1: y_0 = (C_0 . B_0) x_0, state = B_0 (outer) x_0, independent of A and dt
    cb = np.einsum("bthn,bthn->bth", Ct, Bt)
    assert rel_fro(y, cb[..., None] * x) < 1e-14
    assert rel_fro(s, np.einsum("bhn,bhd->bhnd", Bt[:, 0], x[:, 0])) < 1e-14


def impulse_case(T=40, dt_value=0.3, seed=3):
    rng = np.random.default_rng(seed)
    H, N, D = 3, 4, 5
    A = f32c(-rng.uniform(0.05, 0.5, H) + 1j * rng.uniform(0.35, 2.2, H))
    b0 = f32c(rng.standard_normal((H, N)) + 1j * rng.standard_normal((H, N)))
    c0 = f32c(rng.standard_normal((H, N)) + 1j * rng.standard_normal((H, N)))
    x0 = f32c(rng.standard_normal((H, D)) + 1j * rng.standard_normal((H, D)))
    x = np.zeros((1, T, H, D), complex)
    x[0, 0] = x0
    Bt = np.broadcast_to(b0, (1, T, H, N)).copy()
    Ct = np.broadcast_to(c0, (1, T, H, N)).copy()
    dt = np.full((1, T, H), np.float32(dt_value), np.float64)
    return x, A, Bt, Ct, dt, b0, c0, x0


def test_impulse_response_geometric():
    x, A, Bt, Ct, dt, b0, c0, x0 = impulse_case()
    y, _ = run(x, A, Bt, Ct, dt)
    delta = np.log1p(np.exp(np.float64(np.float32(0.3))))
    t = np.arange(x.shape[1])[:, None]
    cb = np.sum(c0 * b0, axis=-1)                               # (H,)
    expect = cb[None, :, None] * np.exp(t[..., None] * delta * A[None, :, None]) * x0[None]
    assert rel_fro(y[0], expect) < 1e-12


def test_dt_zero_gives_power_of_two():
    # softplus(0) = ln 2, so A_bar = exp(ln2 * A) = 2^A; the impulse response is (C.B) 2^(A t) x0
    x, A, Bt, Ct, dt, b0, c0, x0 = impulse_case(dt_value=0.0)
    y, _ = run(x, A, Bt, Ct, dt)
    t = np.arange(x.shape[1])
    cb = np.sum(c0 * b0, axis=-1)
    pw = np.power(2.0 + 0j, t[:, None] * A[None, :])            # (T,H)
    expect = cb[None, :, None] * pw[..., None] * x0[None]
    assert rel_fro(y[0], expect) < 1e-12


def test_scalar_case_is_first_order_iir_filter():
    # N = D = 1 with a constant step: s_t = a s_{t-1} + B_t x_t is scipy's lfilter([1], [1, -a])
    rng = np.random.default_rng(11)
    T = 300
    A = f32c(np.array([-0.2 + 0.9j]))
    x = f32c(rng.standard_normal((1, T, 1, 1)) + 1j * rng.standard_normal((1, T, 1, 1)))
    Bt = f32c(rng.standard_normal((1, T, 1, 1)) + 1j * rng.standard_normal((1, T, 1, 1)))
    Ct = f32c(rng.standard_normal((1, T, 1, 1)) + 1j * rng.standard_normal((1, T, 1, 1)))
    dtv = np.float32(-0.4)
    dt = np.full((1, T, 1), dtv, np.float64)
    y, s = run(x, A, Bt, Ct, dt)
    a = np.exp(np.log1p(np.exp(np.float64(dtv))) * A[0])
    u = Bt[0, :, 0, 0] * x[0, :, 0, 0]
    sf = scipy.signal.lfilter([1.0], [1.0, -a], u)
    assert rel_fro(y[0, :, 0, 0], Ct[0, :, 0, 0] * sf) < 1e-12
    assert abs(s[0, 0, 0, 0] - sf[-1]) < 1e-12 * max(1.0, abs(sf[-1]))


def test_golden_widget_pair_rotation():
    # The landing page's eigen-pair probe prints lambda = 0.642 + 0.518i and theta = 38.8 deg
    # (truncated display of 38.898 deg).
    vals = {}
    with open(os.path.join(GOLDEN, "widget_pair16.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float(v)
    lam = vals["lambda_re"] + 1j * vals["lambda_im"]
    # dt = 0 gives delta = ln 2, so A = log(lambda) / ln 2 makes A_bar = lambda.
    A = np.array([np.log(lam) / np.log(2.0)])
    T = 12
    x = np.zeros((1, T, 1, 1), complex)
    x[0, 0, 0, 0] = 1.0
    ones = np.ones((1, T, 1, 1), complex)
    y, _ = run(x, A, ones, ones, np.zeros((1, T, 1)))
    ratio = y[0, 1:, 0, 0] / y[0, :-1, 0, 0]
    theta = np.degrees(np.angle(ratio))
    assert np.all((theta >= vals["theta_lo_deg"]) & (theta < vals["theta_hi_deg"]))
    assert np.allclose(np.abs(ratio), abs(lam), rtol=1e-6)


def test_linearity_in_x():
    x1, A, Bt, Ct, dt = rand_case(T=50, N=6, D=5, seed=1)
    x2 = rand_case(T=50, N=6, D=5, seed=2)[0]
    a, b = 0.75, -1.5
    y1, s1 = run(x1, A, Bt, Ct, dt)
    y2, s2 = run(x2, A, Bt, Ct, dt)
    y3, s3 = run(f32c(a * x1 + b * x2), A, Bt, Ct, dt)
    # inputs are rounded to complex64 on the way in, so compare at that precision
    assert rel_fro(y3, a * y1 + b * y2) < 1e-6
    assert rel_fro(s3, a * s1 + b * s2) < 1e-6


def test_causality():
    x, A, Bt, Ct, dt = rand_case(T=60, seed=5)
    y, _ = run(x, A, Bt, Ct, dt)
    x2 = x.copy()
    x2[:, 37] += 3.0 - 2.0j
    y2, _ = run(x2, A, Bt, Ct, dt)
    assert np.array_equal(y[:, :37], y2[:, :37])
    assert not np.allclose(y[:, 37:], y2[:, 37:])


def test_head_and_batch_permutation():
    x, A, Bt, Ct, dt = rand_case(Bn=3, T=30, H=4, seed=6)
    y, s = run(x, A, Bt, Ct, dt)
    pb, ph = np.array([2, 0, 1]), np.array([3, 1, 0, 2])
    yp, sp = run(x[pb][:, :, ph], A[ph], Bt[pb][:, :, ph], Ct[pb][:, :, ph], dt[pb][:, :, ph])
    assert np.array_equal(yp, y[pb][:, :, ph])
    assert np.array_equal(sp, s[pb][:, ph])


def test_conjugation_symmetry():
    x, A, Bt, Ct, dt = rand_case(T=40, seed=8)
    y, s = run(x, A, Bt, Ct, dt)
    yc, sc = run(np.conj(x), np.conj(A), np.conj(Bt), np.conj(Ct), dt)
    assert rel_fro(yc, np.conj(y)) < 1e-13
    assert rel_fro(sc, np.conj(s)) < 1e-13


def test_split_continuation():
    x, A, Bt, Ct, dt = rand_case(T=70, seed=9)
    y, s = run(x, A, Bt, Ct, dt)
    t1 = 29
    ya, sa = run(x[:, :t1], A, Bt[:, :t1], Ct[:, :t1], dt[:, :t1])
    yb, sb = run(x[:, t1:], A, Bt[:, t1:], Ct[:, t1:], dt[:, t1:], s0=sa)
    assert rel_fro(np.concatenate([ya, yb], axis=1), y) < 1e-13
    assert rel_fro(sb, s) < 1e-13


def test_real_reduction():
    x, A, Bt, Ct, dt = rand_case(T=40, seed=10)
    y, s = run(x.real, A.real, Bt.real, Ct.real, dt)
    assert np.max(np.abs(y.imag)) == 0.0 and np.max(np.abs(s.imag)) == 0.0
    assert np.linalg.norm(y.real) > 0


def test_output_limit_keeps_state():
    x, A, Bt, Ct, dt = rand_case(T=50, seed=12)
    y, s = run(x, A, Bt, Ct, dt)
    y2, s2 = run(x, A, Bt, Ct, dt, t_y=17)
    assert np.array_equal(y2[:, :17], y[:, :17])
    assert np.all(y2[:, 17:] == 0)
    assert np.array_equal(s2, s)


def test_threads_do_not_change_result():
    x, A, Bt, Ct, dt = rand_case(Bn=3, T=33, H=3, seed=13)
    y1, s1 = run(x, A, Bt, Ct, dt, threads=1)
    y4, s4 = run(x, A, Bt, Ct, dt, threads=4)
    assert np.array_equal(y1, y4) and np.array_equal(s1, s4)


@pytest.mark.parametrize("T,Q", [(64, 1), (64, 2), (64, 16), (64, 64), (70, 16), (50, 64), (96, 32)])
@pytest.mark.parametrize("dt_mode", ["normal", "zero"])
def test_chunk_size_invariance(T, Q, dt_mode):
    # landing page, "03 Chunkwise SSD": chunked and sequential forms agree (< 1e-5 max |diff|)
    x, A, Bt, Ct, dt = rand_case(Bn=2, T=T, H=3, N=8, D=6, seed=T + Q, dt_mode=dt_mode)
    y, s = run(x, A, Bt, Ct, dt)
    yc, sc = chunkwise(x, A, Bt, Ct, dt, Q)
    assert np.max(np.abs(yc - y)) < 1e-10
    assert rel_fro(yc, y) < 1e-12 and rel_fro(sc, s) < 1e-12


def test_skill2_example_shapes():
    # "Skills Reference", Skill 2: B=2, T=16, H=2, D=4, N=4, dt = 0, chunk 4,
    # A = randn - 1 (so Re A may be positive), Re(y) within atol 1e-4.
    rng = np.random.default_rng(0)
    cn = lambda *s: (rng.standard_normal(s) + 1j * rng.standard_normal(s)) / np.sqrt(2)
    x, Bt, Ct = f32c(cn(2, 16, 2, 4)), f32c(cn(2, 16, 2, 4)), f32c(cn(2, 16, 2, 4))
    A = f32c(cn(2) - 1.0)
    dt = np.zeros((2, 16, 2))
    y, _ = run(x, A, Bt, Ct, dt)
    yc, _ = chunkwise(x, A, Bt, Ct, dt, 4)
    assert np.allclose(yc.real, y.real, atol=1e-4)


def test_tiny_workload_finishes_and_is_finite():
    for w in (inputs.TINY, inputs.TINY_DT0):
        inp = inputs.generate(w)
        c = inp.complex()
        y, s = run(c["x"], c["A"], c["B"], c["C"], c["dt"])
        yc, sc = chunkwise(c["x"], c["A"], c["B"], c["C"], c["dt"], w.Q)
        assert np.all(np.isfinite(y)) and np.all(np.isfinite(s))
        assert rel_fro(yc, y) < 1e-12 and rel_fro(sc, s) < 1e-12
