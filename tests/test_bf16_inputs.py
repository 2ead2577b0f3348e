"""BF16 activations (NEXT-2, the bfloat16 half: ssd_complex_fwd_bf16): x, B_t and
C_t in bfloat16, A, dt, the states and y in fp32. The oracle scans the same
bfloat16 values (held exactly in float64), so each comparison measures the
kernel alone, at the TF32 path's tolerance (relative Frobenius error 2e-3 on y
and the final state). What rounding fp32 data to bfloat16 does to the result
belongs to the data, not to the kernel: it is recorded beside the comparisons
(about 3e-3 for these draws) and bounded loosely."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import naive_scan, naive_scan_inputs
from state_space_sequence_complex_gb300 import inputs, ssdc
from tests.gpu_util import RECORDED, assert_close, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from state_space_sequence_complex_gb300 import build
    build.build()
    ssdc.load()


def _bf16(a):
    """float32 array -> the same values rounded to bfloat16 (to nearest even), as float32."""
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).to(torch.float32).numpy()


def bf16_values(inp):
    """The inputs with x, B and C rounded to bfloat16 (A and dt unchanged)."""
    return dataclasses.replace(inp, x_re=_bf16(inp.x_re), x_im=_bf16(inp.x_im), B_re=_bf16(inp.B_re),
                               B_im=_bf16(inp.B_im), C_re=_bf16(inp.C_re), C_im=_bf16(inp.C_im))


def run_bf16(inp, Q, s0=None, real_x=False):
    """The library on bfloat16 copies of x, B, C; returns complex128 (y, final state)."""
    a = inp.arrays()
    dev = lambda k, dt=torch.float32: torch.from_numpy(np.ascontiguousarray(a[k])).cuda().to(dt)
    h = lambda k: dev(k, torch.bfloat16)
    f = ssdc.Forward(*inp.dims, Q, "tf32", bf16_inputs=True)
    kw = {}
    if s0 is not None:
        kw = dict(s0_re=torch.from_numpy(np.ascontiguousarray(s0.real, dtype=np.float32)).cuda(),
                  s0_im=torch.from_numpy(np.ascontiguousarray(s0.imag, dtype=np.float32)).cuda())
    y_re, y_im, fs_re, fs_im = f(h("x_re"), None if real_x else h("x_im"), dev("A_re"), dev("A_im"), h("B_re"),
                                 h("B_im"), h("C_re"), h("C_im"), dev("dt"), **kw)
    torch.cuda.synchronize()
    st = f.status()
    assert st == ssdc.SSDC_OK, ssdc.strerror(st)
    assert ssdc.last_path() == "fused_tmem" and ssdc.last_launch_count() == 1
    y = y_re.double().cpu().numpy() + 1j * y_im.double().cpu().numpy()
    s = fs_re.double().cpu().numpy() + 1j * fs_im.double().cpu().numpy()
    return y, s


# (B, T, H, D, N, Q): the tiny shape, the single-layer shape, feature sizes below the tile,
# every chunk size, ragged tails, several sequences per CTA
CASES = [
    (1, 128, 2, 8, 8, 16),
    (2, 2048, 16, 64, 64, 64),
    (2, 257, 3, 40, 16, 32),
    (2, 64 * 9 + 13, 3, 64, 64, 64),
    (2, 300, 3, 64, 64, 128),
    (2, 511, 3, 24, 56, 256),
    (20, 200, 8, 64, 64, 64),
    (1, 10, 2, 64, 64, 64),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}T{}H{}D{}N{}Q{}".format(*c))
def test_bf16_inputs_match_oracle_on_the_same_values(case):
    Bn, T, H, D, N, Q = case
    inp = inputs.custom(Bn, T, H, D, N, seed=7000 + T + Q)
    hb = bf16_values(inp)
    y_ref, s_ref = naive_scan_inputs(hb)
    y, s = run_bf16(inp, Q)
    assert_close(y, s, y_ref, s_ref, "tf32", "bf16 inputs")
    # the data's own rounding, for reference: the fp32 inputs' scan against the bfloat16 one
    y32, s32 = naive_scan_inputs(inp)
    ey, es = rel_fro(y_ref, y32), rel_fro(s_ref, s32)
    RECORDED.append(("oracle on the bf16 values against the oracle on the fp32 data", "bf16 data",
                     "B{}T{}H{}D{}N{}Q{}".format(*case), ey, es))
    assert ey < 2e-2 and es < 2e-2


def test_bf16_real_x():
    inp = inputs.custom(2, 300, 4, 64, 64, seed=7100)
    hb = bf16_values(inp)
    y_ref, s_ref = naive_scan(hb.x_re, np.zeros_like(hb.x_re), hb.A_re, hb.A_im, hb.B_re, hb.B_im, hb.C_re,
                              hb.C_im, hb.dt)
    y, s = run_bf16(inp, 64, real_x=True)
    assert_close(y, s, y_ref, s_ref, "tf32", "bf16 inputs, real x")


@pytest.mark.parametrize("Q", [64, 128])
def test_bf16_initial_state(Q):
    inp = inputs.custom(3, 330, 5, 64, 64, seed=7200 + Q)
    rng = np.random.default_rng(Q)
    Bn, T, H, N, D = inp.dims
    s0 = 8.0 * np.sqrt(0.5) * (rng.standard_normal((Bn, H, N, D)) + 1j * rng.standard_normal((Bn, H, N, D)))
    s0_32 = s0.real.astype(np.float32).astype(np.float64) + 1j * s0.imag.astype(np.float32).astype(np.float64)
    y_ref, s_ref = naive_scan_inputs(bf16_values(inp), s0=s0_32)
    y, s = run_bf16(inp, Q, s0=s0)
    assert_close(y, s, y_ref, s_ref, "tf32", f"bf16 inputs, initial state, Q={Q}")


def test_bf16_matches_tf32_path_on_the_same_values():
    # the fp32 entry point given the bfloat16 values (exact in fp32) computes the same scan:
    # both within the tolerance of each other (only C B^T is multiplied differently)
    from tests.gpu_util import run_library
    inp = inputs.custom(2, 640, 8, 64, 64, seed=7300)
    hb = bf16_values(inp)
    y16, s16 = run_bf16(inp, 64)
    y32, s32, _ = run_library(hb, 64, "tf32")
    assert rel_fro(y16, y32) <= 2e-3 and rel_fro(s16, s32) <= 2e-3


def test_bf16_rejects_other_precisions():
    inp = inputs.custom(1, 64, 2, 64, 64, seed=1)
    with pytest.raises(ssdc.SSDCError):
        ssdc.Forward(*inp.dims, 64, "fp32", bf16_inputs=True)
