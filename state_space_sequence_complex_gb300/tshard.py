"""Sequence (T) sharding of the forward pass: rank r of a group holds tokens
[T_r, T_{r+1}) of every (b, h) sequence of the batch, and the ranks together
produce the scan of the whole sequences.

The one exchange is the state pass between segments (landing page, "03
Chunkwise SSD", the STATE line, applied to whole segments). A segment scanned
from a zero state ends in S_seg and multiplies an incoming state by its total
decay a_seg = prod_t A_bar_t, so it maps S_in to a_seg S_in + S_seg, and
consecutive segments compose as (a2, S2) o (a1, S1) = (a2 a1, a2 S1 + S2).
Each rank therefore

1. forms its segment's (a_seg, S_seg): S_seg is the state its segment leaves
   from zero, without rows of y (ssd_complex_final_state); rank 0, whose
   segment starts from the zero state, scans it in full instead, and its rows
   are final;
2. all-gathers the (a_seg, S_seg) of every rank (one collective);
3. folds the aggregates of ranks 0 .. r-1, in order, into its incoming state;
4. scans its segment from that state (ranks r > 0) for its rows of y and the
   state after the segment; the last rank's is the sequences' final state.

Every computation runs in the backend: ``LibraryBackend`` calls libssdc
(ssd_complex_fwd / _init, ssd_complex_final_state, ssd_complex_segment_decay,
ssd_complex_state_combine) on the rank's GPU; this module only orders the calls
and moves one flat tensor per rank through the collective. A segment boundary
on a chunk boundary keeps the chunking of the whole sequence.
``forward_segments`` runs the same steps for segments held by one process (no
collective).
"""
from __future__ import annotations


class LibraryBackend:
    """Scans and joins segments with libssdc on the current CUDA device.

    Inputs are dicts of planar float32 CUDA tensors keyed x_re, x_im (or None),
    A_re, A_im, B_re, B_im, C_re, C_im, dt, with a segment's (B, T_seg, H, .)."""

    ORDER = ["x_re", "x_im", "A_re", "A_im", "B_re", "B_im", "C_re", "C_im", "dt"]

    def __init__(self, chunk_size: int, precision: str = "tf32"):
        self.Q = chunk_size
        self.precision = precision

    def _forward(self, seg, s0=None):
        from . import ssdc
        Bn, T, H, N = seg["B_re"].shape
        D = seg["x_re"].shape[-1]
        f = ssdc.Forward(Bn, T, H, N, D, self.Q, self.precision, device=seg["x_re"].device)
        kw = {} if s0 is None else dict(s0_re=s0[0], s0_im=s0[1])
        out = f(*[seg[k] for k in self.ORDER], **kw)
        st = f.status()
        if st != ssdc.SSDC_OK:
            raise ssdc.SSDCError(st, "segment scan")
        return out

    @staticmethod
    def _offsets(shape):
        # the four planes of the flat tensor, each starting on a 16-byte boundary
        Bn, H, N, D = shape
        k = -(-Bn * H // 4) * 4
        m = Bn * H * N * D
        return k, m

    def local(self, seg, rows=True):
        """The segment from zero: its outputs (y_re, y_im, fs_re, fs_im) if ``rows``
        (a full scan), else None (the state alone, ssd_complex_final_state), and its
        aggregate (a_seg, S_seg) as one flat tensor [a_re (B H), a_im (B H), S_re
        (B H N D), S_im (B H N D)], each plane padded to 16 bytes."""
        import torch
        from . import ssdc
        if rows:
            out = self._forward(seg)
            fs_re, fs_im = out[2], out[3]
        else:
            out = None
            Bn, T, H, N = seg["B_re"].shape
            D = seg["x_re"].shape[-1]
            f = ssdc.FinalState(Bn, T, H, N, D, self.Q, self.precision, device=seg["x_re"].device)
            fs_re, fs_im = f(*[seg[k] for k in ("x_re", "x_im", "A_re", "A_im", "B_re", "B_im", "dt")])
            st = f.status()
            if st != ssdc.SSDC_OK:
                raise ssdc.SSDCError(st, "segment state")
        shape = self.state_shape(seg)
        Bn, H = shape[0], shape[1]
        k, m = self._offsets(shape)
        flat = torch.zeros(2 * k + 2 * m, dtype=torch.float32, device=fs_re.device)
        a, s = self.unpack(flat, shape)
        ssdc.ssd_complex_segment_decay(seg["A_re"], seg["A_im"], seg["dt"], a_re=a[0], a_im=a[1])
        s[0].copy_(fs_re)
        s[1].copy_(fs_im)
        return out, flat

    @classmethod
    def unpack(cls, flat, shape):
        Bn, H, N, D = shape
        k, m = cls._offsets(shape)
        a = (flat[:Bn * H].view(Bn, H), flat[k:k + Bn * H].view(Bn, H))
        s = (flat[2 * k:2 * k + m].view(Bn, H, N, D), flat[2 * k + m:2 * k + 2 * m].view(Bn, H, N, D))
        return a, s

    def combine(self, a, s_in, s_add):
        """a s_in + s_add per (b, h); s_in None for a zero state."""
        import torch
        from . import ssdc
        out = (torch.empty_like(s_add[0]), torch.empty_like(s_add[1]))
        ssdc.ssd_complex_state_combine(a[0], a[1], None if s_in is None else s_in[0],
                                       None if s_in is None else s_in[1], s_add[0], s_add[1],
                                       out_re=out[0], out_im=out[1])
        return out

    def rescan(self, seg, s_in):
        """(y_re, y_im, fs_re, fs_im) of the segment from the incoming state."""
        return self._forward(seg, s_in)

    @staticmethod
    def state_shape(seg):
        Bn, T, H, N = seg["B_re"].shape
        return Bn, H, N, seg["x_re"].shape[-1]


def incoming_state(backend, flats, rank, shape):
    """The state entering segment `rank`: the aggregates of segments 0 .. rank-1
    folded in order (None for rank 0: the zero state)."""
    s_in = None
    for r in range(rank):
        a, s = backend.unpack(flats[r], shape)
        s_in = backend.combine(a, s_in, s)
    return s_in


def forward(seg, backend, group=None):
    """The forward pass of this rank's segment of a sequence sharded in time over
    the ranks of `group` (torch.distributed, rank order = time order). Returns
    (y_re, y_im, fs_re, fs_im): this segment's rows of y and the state after it
    (on the last rank, the final state of the whole sequences)."""
    import torch
    import torch.distributed as dist
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    shape = backend.state_shape(seg)
    out, flat = backend.local(seg, rows=rank == 0)
    flats = [torch.empty_like(flat) for _ in range(world)]
    dist.all_gather(flats, flat, group=group)
    if rank == 0:  # the first segment starts from the zero state: its local scan is final
        return out
    return backend.rescan(seg, incoming_state(backend, flats, rank, shape))


def forward_segments(segs, backend):
    """The same steps for consecutive segments held by one process: returns the
    list of per-segment (y_re, y_im, fs_re, fs_im)."""
    shape = backend.state_shape(segs[0])
    local = [backend.local(s, rows=r == 0) for r, s in enumerate(segs)]
    flats = [f for _, f in local]
    return [local[0][0]] + [backend.rescan(s, incoming_state(backend, flats, r, shape))
                            for r, s in enumerate(segs) if r > 0]
