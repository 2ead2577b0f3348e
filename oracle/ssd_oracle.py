"""ctypes front end of the C oracle (``ssd_oracle.c``). TEST INFRASTRUCTURE ONLY.

``naive_scan`` runs the plain O(T) complex128 sequential scan of the page
"Extending -- SSM variants & Triton kernels" (Path A, Step 1) with the
discretisation A_bar = exp(softplus(dt) * A). It returns y (B,T,H,D) and the
final state (B,H,N,D) as complex128 numpy arrays; Re(y) is ``y.real``.
``naive_grad`` runs the adjoint of the same recurrence: the gradients of a
real loss with respect to every input, given the output gradients.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB = os.path.join(_HERE, "libssd_oracle.so")
_lib = None


def oracle_library_path() -> str:
    return _LIB


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, no vector intrinsics, -O2)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        f = lib.ssd_oracle_naive
        fp = ctypes.POINTER(ctypes.c_float)
        dp = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        f.argtypes = [fp] * 9 + [dp, dp] + [i64] * 6 + [dp] * 4 + [ctypes.c_int]
        f.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f32(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _f64(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def naive_scan(x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt, *,
               t_y: int | None = None, s0: np.ndarray | None = None,
               threads: int | None = None):
    """Sequential complex128 scan. Returns ``(y, state)`` (complex128).

    ``t_y`` limits the rows of y that are computed (the state still runs over
    all T; rows t >= t_y are returned as zero). ``s0`` is an optional complex
    initial state (B,H,N,D), used only by the continuation check.
    """
    lib = _load()
    Bn, T, H, D = np.shape(x_re)
    N = np.shape(B_re)[-1]
    keep = []
    ptrs = []
    for a in (x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt):
        arr, p = _f32(a)
        keep.append(arr)
        ptrs.append(p)
    if s0 is not None:
        s0r = np.ascontiguousarray(np.real(s0), dtype=np.float64)
        s0i = np.ascontiguousarray(np.imag(s0), dtype=np.float64)
        assert s0r.shape == (Bn, H, N, D)
        p0r, p0i = _f64(s0r), _f64(s0i)
    else:
        p0r = p0i = ctypes.POINTER(ctypes.c_double)()
    ty = T if t_y is None else int(t_y)
    y_re = np.zeros((Bn, T, H, D), np.float64)
    y_im = np.zeros((Bn, T, H, D), np.float64)
    s_re = np.zeros((Bn, H, N, D), np.float64)
    s_im = np.zeros((Bn, H, N, D), np.float64)
    rc = lib.ssd_oracle_naive(*ptrs, p0r, p0i, Bn, T, H, N, D, ty,
                              _f64(y_re), _f64(y_im), _f64(s_re), _f64(s_im),
                              int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"ssd_oracle_naive failed with status {rc}")
    return y_re + 1j * y_im, s_re + 1j * s_im


def _load_bwd():
    lib = _load()
    f = lib.ssd_oracle_naive_bwd
    if f.argtypes is None:
        fp = ctypes.POINTER(ctypes.c_float)
        dp = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        f.argtypes = [fp] * 9 + [dp, dp] + [fp] * 4 + [i64] * 5 + [dp] * 13 + [ctypes.c_int]
        f.restype = ctypes.c_int
    return lib


def naive_grad(x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt, dy, dfs=None, *,
               s0: np.ndarray | None = None, threads: int | None = None) -> dict:
    """Gradients of the sequential scan for the output gradients ``dy``
    (B,T,H,D complex) and ``dfs`` (B,H,N,D complex, None: zero), by the
    adjoint recurrence in complex128. A complex gradient holds dL/dRe in its
    real part and dL/dIm in its imaginary part. Returns a dict with complex128
    ``dx``, ``dA``, ``dB``, ``dC``, ``ds0``, ``dz`` (the gradient of each token's
    log-decay z_t = softplus(dt_t) A, shape (B,T,H)) and float64 ``ddt``."""
    lib = _load_bwd()
    Bn, T, H, D = np.shape(x_re)
    N = np.shape(B_re)[-1]
    keep, ptrs = [], []
    for a in (x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt):
        arr, p = _f32(a)
        keep.append(arr)
        ptrs.append(p)
    null_d = ctypes.POINTER(ctypes.c_double)()
    null_f = ctypes.POINTER(ctypes.c_float)()
    if s0 is not None:
        s0r = np.ascontiguousarray(np.real(s0), dtype=np.float64)
        s0i = np.ascontiguousarray(np.imag(s0), dtype=np.float64)
        assert s0r.shape == (Bn, H, N, D)
        p0 = [_f64(s0r), _f64(s0i)]
    else:
        p0 = [null_d, null_d]
    gy = [_f32(np.real(dy)), _f32(np.imag(dy))]
    assert gy[0][0].shape == (Bn, T, H, D)
    if dfs is not None:
        gs = [_f32(np.real(dfs)), _f32(np.imag(dfs))]
        assert gs[0][0].shape == (Bn, H, N, D)
    else:
        gs = [(None, null_f), (None, null_f)]
    out = {k: np.zeros(s, np.float64) for k, s in (
        ("dx_re", (Bn, T, H, D)), ("dx_im", (Bn, T, H, D)), ("dA_re", (H,)), ("dA_im", (H,)),
        ("dB_re", (Bn, T, H, N)), ("dB_im", (Bn, T, H, N)), ("dC_re", (Bn, T, H, N)),
        ("dC_im", (Bn, T, H, N)), ("ddt", (Bn, T, H)), ("ds0_re", (Bn, H, N, D)),
        ("ds0_im", (Bn, H, N, D)), ("dz_re", (Bn, T, H)), ("dz_im", (Bn, T, H)))}
    order = ("dx_re", "dx_im", "dA_re", "dA_im", "dB_re", "dB_im", "dC_re", "dC_im", "ddt",
             "ds0_re", "ds0_im", "dz_re", "dz_im")
    rc = lib.ssd_oracle_naive_bwd(*ptrs, *p0, gy[0][1], gy[1][1], gs[0][1], gs[1][1],
                                  Bn, T, H, N, D, *[_f64(out[k]) for k in order],
                                  int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"ssd_oracle_naive_bwd failed with status {rc}")
    return {"dx": out["dx_re"] + 1j * out["dx_im"], "dA": out["dA_re"] + 1j * out["dA_im"],
            "dB": out["dB_re"] + 1j * out["dB_im"], "dC": out["dC_re"] + 1j * out["dC_im"],
            "ddt": out["ddt"], "ds0": out["ds0_re"] + 1j * out["ds0_im"],
            "dz": out["dz_re"] + 1j * out["dz_im"]}


def naive_grad_inputs(inp, dy, dfs=None, **kw) -> dict:
    """``naive_grad`` on an ``inputs.Inputs`` bundle."""
    return naive_grad(inp.x_re, inp.x_im, inp.A_re, inp.A_im, inp.B_re, inp.B_im,
                      inp.C_re, inp.C_im, inp.dt, dy, dfs, **kw)


def naive_scan_inputs(inp, **kw):
    """``naive_scan`` on an ``inputs.Inputs`` bundle."""
    return naive_scan(inp.x_re, inp.x_im, inp.A_re, inp.A_im, inp.B_re, inp.B_im,
                      inp.C_re, inp.C_im, inp.dt, **kw)


def head_mix(y, W):
    """The MIMO head mixer on Re(y) (landing page, "02 MIMO Mixer": a fully
    connected 16 x 16 mixer across the SSM heads, 1024 -> 1024 features = 16
    heads x 64, identity-initialised). Output head g of token t is
        out[b, t, g, d] = sum_h W[g, h] Re(y)[b, t, h, d],
    the same H x H matrix for every feature d. y (B,T,H,D) complex or real,
    W (H,H); returns float64 (B,T,H,D)."""
    y = np.asarray(y)
    W = np.asarray(W, dtype=np.float64)
    return np.einsum("gh,bthd->btgd", W, np.real(y).astype(np.float64))

