"""Double-precision CPU chunkwise form of the complex SSD scan (tests only).

Written from the landing page's "03 Chunkwise SSD" equations, independently of
the oracle and of the CUDA path. It exists to pin the oracle (chunkwise and
sequential forms must agree for every chunk size, the landing page's
"numerical match" claim) and to check the decomposition's readings:

* inclusive in-chunk cumulative sum Acs of the log-decay softplus(dt) * A;
* L[l, s] = exp(Acs[l] - Acs[s]) for l >= s, else 0 (diagonal included);
* Y_diag = (C B^T o L) X inside the chunk;
* chunk state S_loc = B^T (dec o X) with dec[s] = exp(Acs[Q-1] - Acs[s]);
* between chunks S_in[c+1] = exp(Acs[Q-1]) S_in[c] + S_loc[c];
* Y_off = (C o exp(Acs)) S_in[c].

A partial last chunk is padded with zero log-decay and zero x, B, C.
"""
from __future__ import annotations

import numpy as np


def softplus(v):
    return np.logaddexp(0.0, v)


def chunkwise(x, A, Bt, Ct, dt, Q):
    """x (B,T,H,D), A (H,), Bt/Ct (B,T,H,N) complex; dt (B,T,H) real.

    Returns y (B,T,H,D) complex128 and the final state (B,H,N,D).
    """
    Bn, T, H, D = x.shape
    N = Bt.shape[-1]
    nc = -(-T // Q)
    Tp = nc * Q
    alog = softplus(dt.astype(np.float64)) * A[None, None, :]  # (B,T,H)
    pad = Tp - T

    def padt(a):
        if pad == 0:
            return a
        w = [(0, 0)] * a.ndim
        w[1] = (0, pad)
        return np.pad(a, w)

    alog, xp, bp, cp = padt(alog), padt(x), padt(Bt), padt(Ct)
    # (B,H,nc,Q,...) views
    alog = alog.reshape(Bn, nc, Q, H).transpose(0, 3, 1, 2)
    xp = xp.reshape(Bn, nc, Q, H, D).transpose(0, 3, 1, 2, 4)
    bp = bp.reshape(Bn, nc, Q, H, N).transpose(0, 3, 1, 2, 4)
    cp = cp.reshape(Bn, nc, Q, H, N).transpose(0, 3, 1, 2, 4)

    acs = np.cumsum(alog, axis=-1)  # inclusive, (B,H,nc,Q)
    diff = acs[..., :, None] - acs[..., None, :]  # [l, s]
    causal = np.tril(np.ones((Q, Q), dtype=bool))
    Lm = np.where(causal, np.exp(np.where(causal, diff, 0.0)), 0.0)
    G = np.einsum("bhcln,bhcsn->bhcls", cp, bp)
    y_diag = np.einsum("bhcls,bhcsd->bhcld", G * Lm, xp)
    dec = np.exp(acs[..., -1:] - acs)  # (B,H,nc,Q)
    s_loc = np.einsum("bhcsn,bhcs,bhcsd->bhcnd", bp, dec, xp)
    a_c = np.exp(acs[..., -1])  # (B,H,nc)

    y = np.empty_like(y_diag)
    s = np.zeros((Bn, H, N, D), np.complex128)
    for c in range(nc):
        y_off = np.einsum("bhln,bhl,bhnd->bhld", cp[:, :, c], np.exp(acs[:, :, c]), s)
        y[:, :, c] = y_diag[:, :, c] + y_off
        s = a_c[:, :, c, None, None] * s + s_loc[:, :, c]
    y = y.transpose(0, 2, 3, 1, 4).reshape(Bn, Tp, H, D)[:, :T]
    return y, s
