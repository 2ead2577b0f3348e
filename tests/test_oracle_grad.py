"""Pins of the gradient oracle (``naive_grad``) against what the mathematics
fixes, none of them computed by the oracle's own adjoint recurrence:

* central finite differences of the forward oracle (itself pinned in
  ``test_oracle.py``), element by element, on inputs and steps that float32
  holds exactly, extrapolated (Richardson) to fourth order;
* PyTorch autograd (complex128) through an independently written quadratic
  form of the scan (the materialised SSD matrix plus the initial-state term);
* the homogeneity identities: y and the final state are linear in x, in B_t
  and in the initial state together with x = 0, and y is linear in C_t, so the
  loss equals the real inner product of each of these with its gradient;
* the degenerate A = 0 (no decay), where the step size has no effect.

Convention: a complex gradient holds dL/dRe in its real part and dL/dIm in
its imaginary part, for the real loss L = sum Re(conj(gy) y) + Re(conj(gs) s_T).
"""
import numpy as np
import pytest

from oracle import naive_grad, naive_scan
from state_space_sequence_complex_gb300 import inputs

NAMES = ("x_re", "x_im", "A_re", "A_im", "B_re", "B_im", "C_re", "C_im", "dt")


def quantised_case(Bn, T, H, D, N, seed, step=2.0 ** -12):
    """Inputs, output gradients and an initial state rounded to multiples of
    ``step``, so that adding +-2^-8 or +-2^-9 to any element stays exact in
    float32 and the finite differences see exactly the intended step."""
    inp = inputs.custom(Bn, T, H, D, N, seed)
    q = lambda a: (np.round(np.asarray(a, np.float64) / step) * step).astype(np.float32)
    arrs = {k: q(v) for k, v in inp.arrays().items()}
    g = inputs.output_grads(Bn, T, H, D, N, seed + 1)
    s0r, s0i = inputs.initial_state(Bn, H, N, D, seed + 2)
    gy = q(g.dy_re).astype(np.float64) + 1j * q(g.dy_im)
    gs = q(g.dfs_re).astype(np.float64) + 1j * q(g.dfs_im)
    s0 = q(s0r).astype(np.float64) + 1j * q(s0i)
    return arrs, gy, gs, s0


def loss(arrs, gy, gs, s0):
    y, s = naive_scan(*[arrs[k] for k in NAMES], s0=s0, threads=1)
    return float(np.sum(gy.real * y.real + gy.imag * y.imag)
                 + np.sum(gs.real * s.real + gs.imag * s.imag))


def grads(arrs, gy, gs, s0, threads=1):
    return naive_grad(*[arrs[k] for k in NAMES], gy.astype(np.complex64),
                      None if gs is None else gs.astype(np.complex64), s0=s0, threads=threads)


def as_real_grads(g):
    """The oracle's gradients as dL/d(input plane), keyed like the inputs."""
    return {"x_re": g["dx"].real, "x_im": g["dx"].imag, "A_re": g["dA"].real,
            "A_im": g["dA"].imag, "B_re": g["dB"].real, "B_im": g["dB"].imag,
            "C_re": g["dC"].real, "C_im": g["dC"].imag, "dt": g["ddt"],
            "s0_re": g["ds0"].real, "s0_im": g["ds0"].imag}


def fd(fun, h):
    """Fourth-order central difference: Richardson on steps h and 2h."""
    d1 = (fun(h) - fun(-h)) / (2 * h)
    d2 = (fun(2 * h) - fun(-2 * h)) / (4 * h)
    return (4 * d1 - d2) / 3


@pytest.mark.parametrize("shape", [(1, 6, 2, 3, 2), (2, 5, 1, 2, 3)], ids=["B1T6H2D3N2", "B2T5H1D2N3"])
def test_grad_matches_finite_differences(shape):
    Bn, T, H, D, N = shape
    arrs, gy, gs, s0 = quantised_case(Bn, T, H, D, N, seed=11 + T)
    g = as_real_grads(grads(arrs, gy, gs, s0))
    h = 2.0 ** -9
    checked = 0
    for name in NAMES + ("s0_re", "s0_im"):
        shape_ = s0.shape if name.startswith("s0") else arrs[name].shape
        for idx in np.ndindex(*shape_):
            def f(e, name=name, idx=idx):
                a = dict(arrs)
                s = s0
                if name.startswith("s0"):
                    s = s0.copy()
                    s[idx] += e if name == "s0_re" else 1j * e
                else:
                    a[name] = arrs[name].copy()
                    a[name][idx] += np.float32(e)
                return loss(a, gy, gs, s)
            num = fd(f, h)
            assert abs(num - g[name][idx]) <= 2e-8 * (1.0 + abs(num)), (name, idx, num, g[name][idx])
            checked += 1
    assert checked == 2 * Bn * T * H * D + 2 * H + 4 * Bn * T * H * N + Bn * T * H + 2 * Bn * H * N * D


def test_grad_matches_autograd_of_ssd_matrix():
    torch = pytest.importorskip("torch")
    Bn, T, H, D, N = 2, 23, 3, 4, 5
    inp = inputs.custom(Bn, T, H, D, N, seed=21)
    og = inputs.output_grads(Bn, T, H, D, N, seed=22)
    s0r, s0i = inputs.initial_state(Bn, H, N, D, seed=23)
    c = inp.complex()
    leaf = lambda a: torch.tensor(a, dtype=torch.complex128, requires_grad=True)
    x, A, Bt, Ct = leaf(c["x"]), leaf(c["A"]), leaf(c["B"]), leaf(c["C"])
    s0 = leaf(s0r.astype(np.float64) + 1j * s0i)
    dt = torch.tensor(c["dt"], dtype=torch.float64, requires_grad=True)
    # quadratic form: y_t = sum_{s<=t} (C_t . B_s) e^{Lam_t - Lam_s} x_s + e^{Lam_t} C_t s0,
    # s_T = e^{Lam_{T-1}} s0 + sum_s e^{Lam_{T-1} - Lam_s} B_s (outer) x_s
    lam = torch.cumsum(torch.nn.functional.softplus(dt).to(torch.complex128) * A, dim=1)  # (B,T,H)
    diff = lam[:, :, None, :] - lam[:, None, :, :]  # (B,t,s,H)
    causal = torch.tril(torch.ones(T, T, dtype=torch.bool))[None, :, :, None]
    decay = torch.where(causal, torch.exp(torch.where(causal, diff, torch.zeros_like(diff))),
                        torch.zeros_like(diff))
    cb = torch.einsum("bthn,bshn->btsh", Ct, Bt)
    y = torch.einsum("btsh,bshd->bthd", cb * decay, x)
    y = y + torch.exp(lam)[..., None] * torch.einsum("bthn,bhnd->bthd", Ct, s0)
    last = lam[:, -1, :]  # (B,H)
    dec = torch.exp(last[:, None, :] - lam)  # (B,T,H)
    st = torch.exp(last)[..., None, None] * s0 + torch.einsum("bsh,bshn,bshd->bhnd", dec, Bt, x)
    gy = torch.tensor(og.complex()["dy"])
    gs = torch.tensor(og.complex()["dfs"])
    L = (gy.conj() * y).real.sum() + (gs.conj() * st).real.sum()
    L.backward()
    g = naive_grad(*[inp.arrays()[k] for k in NAMES], og.dy_re + 1j * og.dy_im,
                   og.dfs_re + 1j * og.dfs_im, s0=s0r.astype(np.float64) + 1j * s0i)
    pairs = [("dx", x), ("dA", A), ("dB", Bt), ("dC", Ct), ("ds0", s0)]
    for k, t in pairs:
        ref = t.grad.numpy()
        assert np.linalg.norm(g[k] - ref) <= 1e-11 * np.linalg.norm(ref), k
    ref = dt.grad.numpy()
    assert np.linalg.norm(g["ddt"] - ref) <= 1e-11 * np.linalg.norm(ref)

    # dz: the same loss as a function of the per-token log-decays z_t = softplus(dt_t) A
    z = (torch.nn.functional.softplus(dt).to(torch.complex128) * A).detach().requires_grad_(True)
    lam = torch.cumsum(z, dim=1)
    diff = lam[:, :, None, :] - lam[:, None, :, :]
    decay = torch.where(causal, torch.exp(torch.where(causal, diff, torch.zeros_like(diff))),
                        torch.zeros_like(diff))
    y = torch.einsum("btsh,bshd->bthd", cb.detach() * decay, x.detach())
    y = y + torch.exp(lam)[..., None] * torch.einsum("bthn,bhnd->bthd", Ct.detach(), s0.detach())
    last = lam[:, -1, :]
    dec = torch.exp(last[:, None, :] - lam)
    st = (torch.exp(last)[..., None, None] * s0.detach()
          + torch.einsum("bsh,bshn,bshd->bhnd", dec, Bt.detach(), x.detach()))
    ((gy.conj() * y).real.sum() + (gs.conj() * st).real.sum()).backward()
    ref = z.grad.numpy()
    assert np.linalg.norm(g["dz"] - ref) <= 1e-11 * np.linalg.norm(ref)


def test_grad_homogeneity_identities():
    Bn, T, H, D, N = 2, 40, 2, 6, 5
    inp = inputs.custom(Bn, T, H, D, N, seed=31)
    og = inputs.output_grads(Bn, T, H, D, N, seed=32)
    a = inp.arrays()
    gy = og.dy_re.astype(np.float64) + 1j * og.dy_im
    gs = og.dfs_re.astype(np.float64) + 1j * og.dfs_im
    rip = lambda u, v: float(np.sum(u.real * v.real + u.imag * v.imag))  # real inner product
    c = inp.complex()

    y, s = naive_scan(*[a[k] for k in NAMES])
    L = rip(gy, y) + rip(gs, s)
    g = naive_grad(*[a[k] for k in NAMES], gy, gs)
    # y and s_T are linear in x and (separately) in B_t; y alone is linear in C_t
    assert abs(rip(g["dx"], c["x"]) - L) <= 1e-10 * abs(L)
    assert abs(rip(g["dB"], c["B"]) - L) <= 1e-10 * abs(L)
    Ly = rip(gy, y)
    gC = naive_grad(*[a[k] for k in NAMES], gy, None)
    assert abs(rip(gC["dC"], c["C"]) - Ly) <= 1e-10 * abs(Ly)

    # with x = 0 the outputs are linear in the initial state
    s0r, s0i = inputs.initial_state(Bn, H, N, D, seed=33)
    s0 = s0r.astype(np.float64) + 1j * s0i
    a0 = dict(a, x_re=np.zeros_like(a["x_re"]), x_im=np.zeros_like(a["x_im"]))
    y0, st0 = naive_scan(*[a0[k] for k in NAMES], s0=s0)
    L0 = rip(gy, y0) + rip(gs, st0)
    g0 = naive_grad(*[a0[k] for k in NAMES], gy, gs, s0=s0)
    assert abs(rip(g0["ds0"], s0) - L0) <= 1e-10 * abs(L0)


def test_grad_no_decay_and_zero_output_grads():
    Bn, T, H, D, N = 1, 30, 2, 4, 4
    inp = inputs.custom(Bn, T, H, D, N, seed=41)
    og = inputs.output_grads(Bn, T, H, D, N, seed=42)
    a = inp.arrays()
    gy = og.dy_re + 1j * og.dy_im
    gs = og.dfs_re + 1j * og.dfs_im
    # A = 0: A_bar = 1 whatever dt, so dt has no effect on the loss
    a0 = dict(a, A_re=np.zeros_like(a["A_re"]), A_im=np.zeros_like(a["A_im"]))
    g = naive_grad(*[a0[k] for k in NAMES], gy, gs)
    assert np.all(g["ddt"] == 0.0)
    assert np.linalg.norm(g["dx"]) > 0 and np.linalg.norm(g["dA"]) > 0
    # zero output gradients: every input gradient is zero
    g = naive_grad(*[a[k] for k in NAMES], np.zeros_like(gy), np.zeros_like(gs))
    for k in ("dx", "dA", "dB", "dC", "ddt", "ds0"):
        assert np.all(g[k] == 0.0), k


def test_grad_threads_do_not_change_results():
    Bn, T, H, D, N = 3, 17, 4, 4, 3
    inp = inputs.custom(Bn, T, H, D, N, seed=51)
    og = inputs.output_grads(Bn, T, H, D, N, seed=52)
    a = inp.arrays()
    args = [a[k] for k in NAMES] + [og.dy_re + 1j * og.dy_im, og.dfs_re + 1j * og.dfs_im]
    g1 = naive_grad(*args, threads=1)
    g4 = naive_grad(*args, threads=4)
    for k in g1:
        assert np.array_equal(g1[k], g4[k]), k
