"""Error model of the TF32 tensor-core path (tests only): the chunked forward
computed in float64 with the data flow of the fused kernels, where each source
of rounding the kernels add can be switched on alone:

* ``operands``: the operands of the four real-GEMM products (C and B of C B^T;
  P and x of Y_diag; x and dec o B of the chunk state; C' = C o exp(Acs) and
  S_in of Y_off) rounded to TF32 (10 explicit mantissa bits), to nearest with
  ties to even (``"rn"``) or away from zero (``"rna"``, what the kernels do to
  the operands they write), or toward zero (``"rz"``, what the tensor core does
  to an fp32 operand); products and sums stay exact;
* ``acs32``: the in-chunk cumulative log-decay summed in float32 (the kernels'
  producer warp), every decay a float64 exponential of its float32 differences;
* ``exp32``: every decay factor (L, dec, exp(Acs), a_c) rounded to float32 after
  its float64 exponential (a lower bound of the hardware exponentials' error);
* ``state32``: the state pass S_in[c+1] = a_c S_in[c] + S_loc[c] rounded to float32
  at every chunk.

It follows the landing page's "03 Chunkwise SSD" equations (as the chunkwise
reference does) and shares no code with the oracle or the CUDA path. The
relative Frobenius error of each switched-on source against the oracle, and of
all together, shows where the TF32 path's error comes from.
"""
from __future__ import annotations

import numpy as np


def round_tf32(a, mode):
    """Round float32 values to TF32 (drop 13 of the 23 mantissa bits)."""
    if mode is None:
        return a
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32)
    if mode == "rn":  # to nearest, ties to even
        lsb = (u >> 13) & 1
        u = (u + np.uint32(0x0FFF) + lsb) & np.uint32(0xFFFFE000)
    elif mode == "rna":  # to nearest, ties away from zero
        u = (u + np.uint32(0x1000)) & np.uint32(0xFFFFE000)
    elif mode == "rz":
        u = u & np.uint32(0xFFFFE000)
    else:
        raise ValueError(mode)
    return u.view(np.float32).astype(np.float64)


def _rc(z, mode):
    """Complex array with each plane rounded (TF32 of its float32 value)."""
    if mode is None:
        return z
    return round_tf32(z.real.astype(np.float32), mode) + 1j * round_tf32(z.imag.astype(np.float32), mode)


def _f32(z, on):
    if not on:
        return z
    return z.real.astype(np.float32).astype(np.float64) + 1j * z.imag.astype(np.float32).astype(np.float64)


def chunked_forward(x, A, Bt, Ct, dt, Q, operands=None, acs32=False, exp32=False, state32=False,
                    loaded=None, state_op=None):
    """x (B,T,H,D), A (H,), Bt/Ct (B,T,H,N) complex; dt (B,T,H). T a multiple of Q.

    ``loaded`` rounds the two operands that the MMA reads as loaded from memory
    (C and B of C B^T), and ``state_op`` the incoming state of Y_off, which the
    kernels keep in float32 for the state pass, differently from the rest
    (default: as ``operands``)."""
    loaded = operands if loaded is None else loaded
    state_op = operands if state_op is None else state_op
    Bn, T, H, D = x.shape
    N = Bt.shape[-1]
    nc = T // Q
    assert nc * Q == T
    sp = np.logaddexp(0.0, dt.astype(np.float64))
    alog = sp * A[None, None, :]
    alog = alog.reshape(Bn, nc, Q, H).transpose(0, 3, 1, 2)  # (B,H,nc,Q)
    xp = x.reshape(Bn, nc, Q, H, D).transpose(0, 3, 1, 2, 4)
    bp = Bt.reshape(Bn, nc, Q, H, N).transpose(0, 3, 1, 2, 4)
    cp = Ct.reshape(Bn, nc, Q, H, N).transpose(0, 3, 1, 2, 4)
    if acs32:
        a32 = alog.real.astype(np.float32) + 1j * alog.imag.astype(np.float32)
        acs = np.cumsum(a32, axis=-1).astype(np.complex64).astype(np.complex128)
    else:
        acs = np.cumsum(alog, axis=-1)
    causal = np.tril(np.ones((Q, Q), dtype=bool))
    diff = acs[..., :, None] - acs[..., None, :]
    Lm = np.where(causal, _f32(np.exp(np.where(causal, diff, 0.0)), exp32), 0.0)
    dec = _f32(np.exp(acs[..., -1:] - acs), exp32)
    eacs = _f32(np.exp(acs), exp32)
    a_c = _f32(np.exp(acs[..., -1]), exp32)

    G = np.einsum("bhcln,bhcsn->bhcls", _rc(cp, loaded), _rc(bp, loaded))
    P = G * Lm
    y_diag = np.einsum("bhcls,bhcsd->bhcld", _rc(P, operands), _rc(xp, operands))
    s_loc = np.einsum("bhcsn,bhcsd->bhcnd", _rc(bp * dec[..., None], operands), _rc(xp, operands))
    cpr = _rc(cp * eacs[..., None], operands)

    y = np.empty_like(y_diag)
    s = np.zeros((Bn, H, N, D), np.complex128)
    for c in range(nc):
        y[:, :, c] = y_diag[:, :, c] + np.einsum("bhln,bhnd->bhld", cpr[:, :, c], _rc(s, state_op))
        s = _f32(a_c[:, :, c, None, None] * s + s_loc[:, :, c], state32)
    y = y.transpose(0, 2, 3, 1, 4).reshape(Bn, T, H, D)
    return y, s
