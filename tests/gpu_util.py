"""Helpers of the GPU parity tests: run the library through the C ABI on the
seeded inputs and compare with the oracle by relative Frobenius error."""
import os

import numpy as np

from state_space_sequence_complex_gb300 import ssdc

# (test, precision, what, rel_fro y, rel_fro state) of every comparison made
# through assert_close; conftest prints them at the end of the session.
RECORDED = []

# Tolerances on relative Frobenius error, y and final state (exact fp32 SIMT
# path and TF32 tensor-core path).
TOL = {"fp32": 1e-5, "tf32": 2e-3, "tf32_staged": 2e-3, "tf32 bwd": 2e-3}


def rel_fro(a, b):
    return float(np.linalg.norm((a - b).ravel()) / max(np.linalg.norm(np.ravel(b)), 1e-300))


def to_device(inp):
    import torch
    return {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in inp.arrays().items()}


def run_library(inp, Q, precision, dev=None, forward=None):
    """Returns (y complex128 numpy, final state complex128 numpy, Forward)."""
    import torch
    t = dev if dev is not None else to_device(inp)
    Bn, T, H, N, D = inp.dims
    f = forward or ssdc.Forward(Bn, T, H, N, D, Q, precision)
    y_re, y_im, fs_re, fs_im = f(t["x_re"], t["x_im"], t["A_re"], t["A_im"], t["B_re"], t["B_im"],
                                 t["C_re"], t["C_im"], t["dt"])
    torch.cuda.synchronize()
    st = f.status()
    assert st == ssdc.SSDC_OK, ssdc.strerror(st)
    y = y_re.double().cpu().numpy() + 1j * y_im.double().cpu().numpy()
    s = fs_re.double().cpu().numpy() + 1j * fs_im.double().cpu().numpy()
    return y, s, f


def assert_close(y, s, y_ref, s_ref, precision, what=""):
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(s)), f"non-finite output {what}"
    ey, es = rel_fro(y, y_ref), rel_fro(s, s_ref)
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    RECORDED.append((test, precision, what, ey, es))
    tol = TOL[precision]
    assert ey <= tol and es <= tol, f"{what} {precision}: rel_fro y {ey:.3e} state {es:.3e} > {tol}"
    return ey, es
