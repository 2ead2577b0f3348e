"""Seeded synthetic inputs for the complex chunkwise SSD forward.

This module is shared by the tests, the bench and the oracle checks. It holds
random draws and shapes only, none of the scan's arithmetic.

Value distributions follow the pages' model ("Mamba-3-Lite" landing page,
"Complex SSD eigenvalue spectrum explorer": decay range alpha in [-3.0, -0.05],
phase velocity omega in [0.35, 2.20]; production shape H=16, D=64, N=64
complex, ctx 2048, chunk 64):

* x, B_t, C_t: complex, real and imaginary parts i.i.d. N(0, 1/2);
* A[h]: Re ~ U[re_lo, re_hi], Im = +-U[0.35, 2.20] with a fair-coin sign;
* dt[b, t, h]: real, N(dt_mean, dt_std), or identically zero.

Draw order is A, dt, x, B_t, C_t from ``numpy.random.default_rng(seed)``
(PCG64). Everything is returned as planar float32 (separate real and
imaginary planes), the layout the library takes.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, chunk size and value distributions."""

    name: str
    B: int
    T: int
    H: int
    D: int
    N: int
    Q: int
    seed: int
    dt_mode: str = "normal"  # "normal" or "zero"
    dt_mean: float = 0.0
    dt_std: float = 1.0
    re_lo: float = -3.0
    re_hi: float = -0.05
    layers: int = 1

    @property
    def token_heads(self) -> int:
        return self.B * self.T * self.H

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the benchmark plan (sizes named by what they are).
TINY = Workload("tiny B1 T128 H2 D8 N8 Q16", 1, 128, 2, 8, 8, 16, seed=0)
TINY_DT0 = TINY.with_(name="tiny B1 T128 H2 D8 N8 Q16 dt=0", dt_mode="zero")
LAYER = Workload("single layer B2 T2048 H16 D64 N64 Q64", 2, 2048, 16, 64, 64, 64, seed=1)
TRAIN28 = Workload("training batch B16 T2048 H16 D64 N64 Q64 x28 layers",
                   16, 2048, 16, 64, 64, 64, seed=200, layers=28)
QSWEEP = Workload("chunk sweep B32 T8192 H16 D64 N64", 32, 8192, 16, 64, 64, 64, seed=3)
LONG = Workload("long memory B4 T65536 H16 D64 N64 Q64", 4, 65536, 16, 64, 64, 64,
                seed=4, dt_mean=-2.0, dt_std=0.5, re_lo=-0.1, re_hi=-0.01)

ALL = {"tiny": TINY, "tiny_dt0": TINY_DT0, "layer": LAYER, "train28": TRAIN28,
       "qsweep": QSWEEP, "long": LONG}


@dataclasses.dataclass
class Inputs:
    """Planar float32 inputs. Shapes: x (B,T,H,D), A (H,), Bt/Ct (B,T,H,N), dt (B,T,H)."""

    x_re: np.ndarray
    x_im: np.ndarray
    A_re: np.ndarray
    A_im: np.ndarray
    B_re: np.ndarray
    B_im: np.ndarray
    C_re: np.ndarray
    C_im: np.ndarray
    dt: np.ndarray

    @property
    def dims(self):
        Bn, T, H, D = self.x_re.shape
        return Bn, T, H, self.B_re.shape[-1], D

    def arrays(self):
        return dict(x_re=self.x_re, x_im=self.x_im, A_re=self.A_re, A_im=self.A_im,
                    B_re=self.B_re, B_im=self.B_im, C_re=self.C_re, C_im=self.C_im,
                    dt=self.dt)

    def complex(self):
        """complex128 views for checks written with complex arithmetic."""
        c = lambda r, i: r.astype(np.float64) + 1j * i.astype(np.float64)
        return dict(x=c(self.x_re, self.x_im), A=c(self.A_re, self.A_im),
                    B=c(self.B_re, self.B_im), C=c(self.C_re, self.C_im),
                    dt=self.dt.astype(np.float64))


def _cnormal_planes(rng, shape):
    s = math.sqrt(0.5)
    re = rng.standard_normal(shape, dtype=np.float32)
    re *= np.float32(s)
    im = rng.standard_normal(shape, dtype=np.float32)
    im *= np.float32(s)
    return re, im


def generate(w: Workload, layer: int = 0, T: int | None = None, B: int | None = None) -> Inputs:
    """Draw the inputs of workload ``w`` (layer ``layer`` uses seed + layer).

    ``T``/``B`` override the sequence length / batch for reduced cases; the
    draws of the per-head A come first, so A does not depend on them.
    """
    Bn = w.B if B is None else B
    Tn = w.T if T is None else T
    rng = np.random.default_rng(w.seed + layer)
    H, D, N = w.H, w.D, w.N
    A_re = rng.uniform(w.re_lo, w.re_hi, H).astype(np.float32)
    mag = rng.uniform(0.35, 2.20, H)
    sign = np.where(rng.integers(0, 2, H) == 1, 1.0, -1.0)
    A_im = (mag * sign).astype(np.float32)
    if w.dt_mode == "zero":
        dt = np.zeros((Bn, Tn, H), np.float32)
    else:
        dt = rng.standard_normal((Bn, Tn, H), dtype=np.float32)
        dt *= np.float32(w.dt_std)
        dt += np.float32(w.dt_mean)
    x_re, x_im = _cnormal_planes(rng, (Bn, Tn, H, D))
    B_re, B_im = _cnormal_planes(rng, (Bn, Tn, H, N))
    C_re, C_im = _cnormal_planes(rng, (Bn, Tn, H, N))
    return Inputs(x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt)


def custom(Bn, T, H, D, N, seed, dt_mode="normal", dt_mean=0.0, dt_std=1.0,
           re_lo=-3.0, re_hi=-0.05) -> Inputs:
    """Inputs of an arbitrary shape with the standard distributions."""
    w = Workload("custom", Bn, T, H, D, N, 1, seed, dt_mode, dt_mean, dt_std, re_lo, re_hi)
    return generate(w)


@dataclasses.dataclass
class OutputGrads:
    """Planar float32 gradients of a loss with respect to the outputs:
    dy (B,T,H,D) and d_final_state (B,H,N,D). A complex gradient holds
    dL/dRe in its real plane and dL/dIm in its imaginary plane."""

    dy_re: np.ndarray
    dy_im: np.ndarray
    dfs_re: np.ndarray
    dfs_im: np.ndarray

    def complex(self):
        c = lambda r, i: r.astype(np.float64) + 1j * i.astype(np.float64)
        return dict(dy=c(self.dy_re, self.dy_im), dfs=c(self.dfs_re, self.dfs_im))


def output_grads(Bn, T, H, D, N, seed) -> OutputGrads:
    """Output gradients with i.i.d. N(0, 1/2) real and imaginary parts, drawn
    dy first, then d_final_state, from ``default_rng(seed)``."""
    rng = np.random.default_rng(seed)
    dy_re, dy_im = _cnormal_planes(rng, (Bn, T, H, D))
    dfs_re, dfs_im = _cnormal_planes(rng, (Bn, H, N, D))
    return OutputGrads(dy_re, dy_im, dfs_re, dfs_im)


def initial_state(Bn, H, N, D, seed) -> tuple[np.ndarray, np.ndarray]:
    """A planar float32 initial state (B,H,N,D), i.i.d. N(0, 1/2) parts."""
    return _cnormal_planes(np.random.default_rng(seed), (Bn, H, N, D))
