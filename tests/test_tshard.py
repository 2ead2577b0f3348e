"""Sequence (T) sharding of the forward pass (state_space_sequence_complex_gb300.tshard):
each rank scans its time segment from zero, the ranks all-gather the segments'
(total decay, end state), each folds the segments before it into its incoming
state and scans its segment from that state.

CPU: gloo ranks (2 and 3) run the exchange logic with an oracle backend (the
complex128 scan of the oracle, and the decay and combine written from their
definitions) and must give the whole-sequence oracle's rows of y and final
state. GPU: the library backend (libssdc's scan, segment decay and state
combine kernels) on segments held by one process, against the oracle; and the
two joining kernels against their definitions."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

SHAPE = dict(Bn=2, T=300, H=3, D=8, N=8)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleBackend:
    """The backend interface of tshard on numpy inputs: scans from the oracle,
    the segment decay exp(sum softplus(dt) A) and the combine a s_in + s_add
    written from their definitions, aggregates flattened into one float64 tensor."""

    def __init__(self):
        from oracle import naive_scan
        self.scan = naive_scan

    def _run(self, seg, s0=None):
        return self.scan(seg["x_re"], seg["x_im"], seg["A_re"], seg["A_im"], seg["B_re"], seg["B_im"],
                         seg["C_re"], seg["C_im"], seg["dt"], s0=s0, threads=1)

    def local(self, seg, rows=True):
        y, s = self._run(seg)
        sp = np.logaddexp(0.0, seg["dt"].astype(np.float64)).sum(axis=1)  # (B, H)
        a = np.exp(sp * (seg["A_re"].astype(np.float64) + 1j * seg["A_im"].astype(np.float64)))
        flat = torch.from_numpy(np.concatenate([a.real.ravel(), a.imag.ravel(), s.real.ravel(), s.imag.ravel()]))
        return ((y, s) if rows else None), flat

    @staticmethod
    def unpack(flat, shape):
        Bn, H, N, D = shape
        v = flat.numpy()
        k, m = Bn * H, Bn * H * N * D
        a = (v[:k] + 1j * v[k:2 * k]).reshape(Bn, H)
        s = (v[2 * k:2 * k + m] + 1j * v[2 * k + m:]).reshape(Bn, H, N, D)
        return a, s

    @staticmethod
    def combine(a, s_in, s_add):
        return s_add if s_in is None else a[:, :, None, None] * s_in + s_add

    def rescan(self, seg, s_in):
        return self._run(seg, s0=s_in)

    @staticmethod
    def state_shape(seg):
        Bn, T, H, N = seg["B_re"].shape
        return Bn, H, N, seg["x_re"].shape[-1]


def _problem():
    from state_space_sequence_complex_gb300 import inputs
    return inputs.custom(SHAPE["Bn"], SHAPE["T"], SHAPE["H"], SHAPE["D"], SHAPE["N"], seed=951)


def _segment(inp, t0, t1):
    return {k: (v if v.ndim == 1 else np.ascontiguousarray(v[:, t0:t1])) for k, v in inp.arrays().items()}


def _bounds(T, world):
    # segment boundaries on multiples of 64 where possible, the last segment takes the rest
    step = max(64, (T // world) // 64 * 64)
    return [min(T, r * step) for r in range(world)] + [T]


def _worker(rank, world, port, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    from state_space_sequence_complex_gb300 import tshard
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        inp = _problem()
        b = _bounds(SHAPE["T"], world)
        y, s = tshard.forward(_segment(inp, b[rank], b[rank + 1]), OracleBackend())
        out[rank] = (y, s)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_sequence_sharded_over_gloo_ranks(world):
    from oracle import naive_scan_inputs
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    inp = _problem()
    y_ref, s_ref = naive_scan_inputs(inp, threads=1)
    b = _bounds(SHAPE["T"], world)
    y = np.concatenate([out[r][0] for r in range(world)], axis=1)
    rel = lambda a, r: np.linalg.norm(a - r) / np.linalg.norm(r)
    assert y.shape == y_ref.shape
    assert rel(y, y_ref) < 1e-12
    assert rel(out[world - 1][1], s_ref) < 1e-12
    # every rank's state is the state after its segment
    for r in range(world - 1):
        _, s_mid = naive_scan_inputs(inputs_prefix(inp, b[r + 1]), threads=1)
        assert rel(out[r][1], s_mid) < 1e-12


def inputs_prefix(inp, t1):
    from state_space_sequence_complex_gb300 import inputs
    return inputs.Inputs(**_segment(inp, 0, t1))


def test_fold_order_and_zero_state():
    be = OracleBackend()
    rng = np.random.default_rng(3)
    shape = (1, 2, 3, 4)
    a1, a2 = rng.standard_normal((1, 2)) + 1j * rng.standard_normal((1, 2)), \
        rng.standard_normal((1, 2)) + 1j * rng.standard_normal((1, 2))
    s1, s2 = (rng.standard_normal(shape) + 1j * rng.standard_normal(shape) for _ in range(2))
    pack = lambda a, s: torch.from_numpy(np.concatenate([a.real.ravel(), a.imag.ravel(), s.real.ravel(),
                                                        s.imag.ravel()]))
    from state_space_sequence_complex_gb300 import tshard
    flats = [pack(a1, s1), pack(a2, s2), None]
    assert tshard.incoming_state(be, flats, 0, shape) is None
    assert np.allclose(tshard.incoming_state(be, flats, 1, shape), s1)
    assert np.allclose(tshard.incoming_state(be, flats, 2, shape), a2[:, :, None, None] * s1 + s2)


# ---------------------------------------------------------------- GPU
@pytest.fixture(scope="module")
def lib():
    from state_space_sequence_complex_gb300 import build, ssdc
    build.build()
    return ssdc.load()


@pytest.mark.gpu
@pytest.mark.parametrize("precision,Q,bounds", [("fp32", 64, [0, 128, 256, 300]), ("tf32", 64, [0, 192, 300]),
                                                ("tf32", 32, [0, 96, 160, 300]), ("fp32", 16, [0, 48, 300])])
def test_library_segments_match_the_oracle(precision, Q, bounds, lib):
    from oracle import naive_scan_inputs
    from state_space_sequence_complex_gb300 import tshard
    from tests.gpu_util import TOL, rel_fro
    inp = _problem()
    y_ref, s_ref = naive_scan_inputs(inp, threads=1)
    segs = []
    for t0, t1 in zip(bounds[:-1], bounds[1:]):
        segs.append({k: torch.from_numpy(v).cuda() for k, v in _segment(inp, t0, t1).items()})
    outs = tshard.forward_segments(segs, tshard.LibraryBackend(Q, precision))
    torch.cuda.synchronize()
    c = lambda re, im: re.double().cpu().numpy() + 1j * im.double().cpu().numpy()
    y = np.concatenate([c(o[0], o[1]) for o in outs], axis=1)
    s = c(outs[-1][2], outs[-1][3])
    assert rel_fro(y, y_ref) <= TOL[precision] and rel_fro(s, s_ref) <= TOL[precision]


@pytest.mark.gpu
def test_joining_kernels(lib):
    from state_space_sequence_complex_gb300 import ssdc
    rng = np.random.default_rng(7)
    Bn, T, H, N, D = 3, 1000, 5, 8, 16
    dt = rng.standard_normal((Bn, T, H)).astype(np.float32)
    A = (-rng.uniform(0.05, 3.0, H) + 1j * rng.uniform(0.35, 2.2, H) * rng.choice([-1, 1], H)) * 1e-3
    A_re, A_im = A.real.astype(np.float32), A.imag.astype(np.float32)
    cu = lambda v: torch.from_numpy(np.ascontiguousarray(v)).cuda()
    a_re, a_im = torch.empty(Bn, H, device="cuda"), torch.empty(Bn, H, device="cuda")
    ssdc.ssd_complex_segment_decay(cu(A_re), cu(A_im), cu(dt), a_re=a_re, a_im=a_im)
    sp = np.logaddexp(0.0, dt.astype(np.float64)).sum(axis=1)
    ref = np.exp(sp * (A_re.astype(np.float64) + 1j * A_im.astype(np.float64)))
    got = a_re.double().cpu().numpy() + 1j * a_im.double().cpu().numpy()
    assert np.max(np.abs(got - ref) / np.abs(ref)) < 1e-6
    # combine, out of place and in place (s_out = s_add), and with a zero incoming state
    shape = (Bn, H, N, D)
    s_in = (rng.standard_normal(shape) + 1j * rng.standard_normal(shape)).astype(np.complex64)
    s_add = (rng.standard_normal(shape) + 1j * rng.standard_normal(shape)).astype(np.complex64)
    av = got.astype(np.complex64)
    exp_out = av[:, :, None, None] * s_in + s_add
    o_re, o_im = torch.empty(shape, device="cuda"), torch.empty(shape, device="cuda")
    ssdc.ssd_complex_state_combine(cu(av.real), cu(av.imag), cu(s_in.real), cu(s_in.imag), cu(s_add.real),
                                   cu(s_add.imag), out_re=o_re, out_im=o_im)
    out = o_re.double().cpu().numpy() + 1j * o_im.double().cpu().numpy()
    assert np.max(np.abs(out - exp_out)) < 1e-5
    add_re, add_im = cu(s_add.real), cu(s_add.imag)
    ssdc.ssd_complex_state_combine(cu(av.real), cu(av.imag), None, None, add_re, add_im, out_re=add_re,
                                   out_im=add_im)
    assert np.array_equal(add_re.cpu().numpy() + 1j * add_im.cpu().numpy(), s_add)
