"""Seeded random problems over the whole supported space, against the oracle.

The other parity tests pick their edge cases by hand; these draw them: 36
problems with B in [1, 4], T in [1, 700], H in [1, 20], N and D multiples of
8 in [8, 64], Q in {16, 32, 64, 128, 256}, a real x or a complex one, an
initial state or none, and sometimes fewer sequences than SMs at Q = N = D =
64 (where the cluster kernel runs). Each runs the TF32 forward (whichever
fused kernel the library picks), the final state alone, and every fourth the
exact fp32 forward and the bfloat16-input forward, each against the oracle's
scan at the path's tolerance (relative Frobenius error on y and the final
state; the bfloat16 path against the oracle on the same bfloat16 values).
Then 24 random problems for the TF32 backward against the gradient oracle."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import naive_scan_inputs
from state_space_sequence_complex_gb300 import inputs, ssdc
from tests.gpu_util import assert_close, to_device

pytestmark = pytest.mark.gpu

ORDER = ["x_re", "x_im", "A_re", "A_im", "B_re", "B_im", "C_re", "C_im", "dt"]
NCASES = 36


@pytest.fixture(scope="module", autouse=True)
def built():
    from state_space_sequence_complex_gb300 import build
    build.build()
    ssdc.load()


def draw(i):
    rng = np.random.default_rng(10_000 + i)
    if i % 6 == 5:  # the cluster kernel's sizes, few sequences
        Bn, H, N, D, Q = int(rng.integers(1, 3)), int(rng.integers(1, 9)), 64, 64, 64
    else:
        Bn, H = int(rng.integers(1, 5)), int(rng.integers(1, 21))
        N, D = 8 * int(rng.integers(1, 9)), 8 * int(rng.integers(1, 9))
        Q = int(rng.choice([16, 32, 64, 128, 256]))
    T = int(rng.integers(1, 701))
    real_x = bool(rng.random() < 0.3)
    with_s0 = bool(rng.random() < 0.4)
    return Bn, T, H, D, N, Q, real_x, with_s0


def cplx(re, im):
    return re.double().cpu().numpy() + 1j * im.double().cpu().numpy()


@pytest.mark.parametrize("i", range(NCASES))
def test_random_problem(i):
    Bn, T, H, D, N, Q, real_x, with_s0 = draw(i)
    what = f"random #{i}: B{Bn} T{T} H{H} D{D} N{N} Q{Q}" + (" real x" if real_x else "") + (" s0" if with_s0 else "")
    inp = inputs.custom(Bn, T, H, D, N, seed=20_000 + i)
    if real_x:
        inp = dataclasses.replace(inp, x_im=np.zeros_like(inp.x_im))
    s0 = None
    kw = {}
    if with_s0:
        rng = np.random.default_rng(30_000 + i)
        s0c = 4.0 * (rng.standard_normal((Bn, H, N, D)) + 1j * rng.standard_normal((Bn, H, N, D)))
        s0 = s0c.real.astype(np.float32) + 1j * s0c.imag.astype(np.float32)
        kw = dict(s0_re=torch.from_numpy(np.ascontiguousarray(s0.real)).cuda(),
                  s0_im=torch.from_numpy(np.ascontiguousarray(s0.imag)).cuda())
    y_ref, s_ref = naive_scan_inputs(inp, s0=None if s0 is None else s0.astype(np.complex128))
    t = to_device(inp)
    if real_x:
        t["x_im"] = None
    # the TF32 forward
    f = ssdc.Forward(Bn, T, H, N, D, Q, "tf32")
    y_re, y_im, fs_re, fs_im = f(*[t[k] for k in ORDER], **kw)
    torch.cuda.synchronize()
    assert f.status() == ssdc.SSDC_OK
    assert ssdc.last_path() in ("fused_tmem", "fused_cluster")
    assert_close(cplx(y_re, y_im), cplx(fs_re, fs_im), y_ref, s_ref, "tf32", what)
    # the final state alone
    g = ssdc.FinalState(Bn, T, H, N, D, Q, "tf32")
    gs_re, gs_im = g(*[t[k] for k in ("x_re", "x_im", "A_re", "A_im", "B_re", "B_im", "dt")], **kw)
    torch.cuda.synchronize()
    assert g.status() == ssdc.SSDC_OK
    s = cplx(gs_re, gs_im)
    assert_close(s, s, s_ref, s_ref, "tf32", what + ", final state alone")
    if i % 4 == 0:  # the exact fp32 forward
        e = ssdc.Forward(Bn, T, H, N, D, Q, "fp32")
        ey_re, ey_im, es_re, es_im = e(*[t[k] for k in ORDER], **kw)
        torch.cuda.synchronize()
        assert e.status() == ssdc.SSDC_OK
        assert_close(cplx(ey_re, ey_im), cplx(es_re, es_im), y_ref, s_ref, "fp32", what + ", exact")
    if i % 4 == 1:  # bfloat16 x, B_t, C_t against the oracle on the same values
        to16 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16)
        hb = dataclasses.replace(inp, **{k: to16(getattr(inp, k)).float().numpy()
                                         for k in ("x_re", "x_im", "B_re", "B_im", "C_re", "C_im")})
        yb_ref, sb_ref = naive_scan_inputs(hb, s0=None if s0 is None else s0.astype(np.complex128))
        tb = dict(t)
        for k in ("x_re", "x_im", "B_re", "B_im", "C_re", "C_im"):
            if tb[k] is not None:
                tb[k] = tb[k].to(torch.bfloat16)
        h = ssdc.Forward(Bn, T, H, N, D, Q, "tf32", bf16_inputs=True)
        hy_re, hy_im, hs_re, hs_im = h(*[tb[k] for k in ORDER], **kw)
        torch.cuda.synchronize()
        assert h.status() == ssdc.SSDC_OK
        assert_close(cplx(hy_re, hy_im), cplx(hs_re, hs_im), yb_ref, sb_ref, "tf32", what + ", bf16 inputs")


NBWD = 24


@pytest.mark.parametrize("i", range(NBWD))
def test_random_backward_problem(i):
    """The TF32 backward on seeded random problems: B in [1, 4], T in [1, 900], H in [1, 19],
    N and D multiples of 8 in [8, 64], Q in {16, 32, 64, 128, 256}, a real x or a complex one,
    a complex loss or one of Re(y) alone, a final-state gradient or none; against the gradient
    oracle at the TF32 bar."""
    from tests.test_backward_gpu import oracle_grads, run_bwd
    from tests.test_backward_tf32_gpu import check_tf32
    rng = np.random.default_rng(40_000 + i)
    Bn, H = int(rng.integers(1, 5)), int(rng.integers(1, 20))
    N, D = 8 * int(rng.integers(1, 9)), 8 * int(rng.integers(1, 9))
    Q = int(rng.choice([16, 32, 64, 128, 256]))
    T = int(rng.integers(1, 901))
    real_x, dy_imag, with_dfs = bool(rng.random() < 0.25), bool(rng.random() < 0.8), bool(rng.random() < 0.7)
    what = f"random backward #{i}: B{Bn} T{T} H{H} D{D} N{N} Q{Q}" + (" real x" if real_x else "") + \
        ("" if dy_imag else ", Re(y) loss") + ("" if with_dfs else ", no final-state gradient")
    inp = inputs.custom(Bn, T, H, D, N, seed=41_000 + i)
    og = inputs.output_grads(Bn, T, H, D, N, seed=42_000 + i)
    b = ssdc.Backward(Bn, T, H, N, D, Q, precision="tf32")
    got = run_bwd(inp, og, Q, backward=b, real_x=real_x, dy_imag=dy_imag, with_dfs=with_dfs)
    ref = oracle_grads(inp, og, real_x=real_x, dy_imag=dy_imag, with_dfs=with_dfs)
    check_tf32(got, ref, inp, what)
