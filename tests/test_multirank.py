"""The bench's multi-rank logic on CPU with two gloo ranks: each rank gets its
own independently seeded batch, and timings are reduced by max over ranks. And
the forward pass sharded over batch rows: each rank scans its rows of one
batch (the oracle's scan), and the rows gathered from every rank are the
whole batch's scan, y and final state, bit for bit (sequences are
independent: no collective on the data path)."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    from state_space_sequence_complex_gb300 import inputs
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks([1.0 + rank, 10.0 * rank, -rank])
        w = inputs.LAYER.with_(T=64, B=1)
        inp = inputs.generate(w, layer=bench.rank_layer(rank))
        digest = float(np.sum(inp.x_re[0, :4, 0, :4]))
        gathered = [None] * world
        dist.all_gather_object(gathered, digest)
        out[rank] = (got, gathered)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    for rank in range(2):
        got, gathered = out[rank]
        assert got == [2.0, 10.0, 0.0]
        assert gathered[0] != gathered[1]  # independent batches per rank


def _rows_worker(rank, world, port, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    from oracle import naive_scan
    from state_space_sequence_complex_gb300 import inputs
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        inp = inputs.custom(4, 130, 3, 8, 8, seed=960)
        rows = slice(rank * 2, rank * 2 + 2)  # rank r holds batch rows 2r, 2r + 1
        a = {k: (v if v.ndim == 1 else np.ascontiguousarray(v[rows])) for k, v in inp.arrays().items()}
        y, s = naive_scan(a["x_re"], a["x_im"], a["A_re"], a["A_im"], a["B_re"], a["B_im"], a["C_re"],
                          a["C_im"], a["dt"], threads=1)
        mine = torch.from_numpy(np.concatenate([y.real.ravel(), y.imag.ravel(), s.real.ravel(), s.imag.ravel()]))
        gathered = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(gathered, mine)
        out[rank] = [g.numpy() for g in gathered]
    finally:
        dist.destroy_process_group()


def test_forward_sharded_over_batch_rows():
    from oracle import naive_scan_inputs
    from state_space_sequence_complex_gb300 import inputs
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rows_worker, args=(2, port, out), nprocs=2, join=True)
    inp = inputs.custom(4, 130, 3, 8, 8, seed=960)
    y_ref, s_ref = naive_scan_inputs(inp, threads=1)
    ny, ns = 2 * 130 * 3 * 8, 2 * 3 * 8 * 8
    for rank in range(2):
        parts = out[rank]
        y = np.concatenate([(p[:ny] + 1j * p[ny:2 * ny]).reshape(2, 130, 3, 8) for p in parts])
        s = np.concatenate([(p[2 * ny:2 * ny + ns] + 1j * p[2 * ny + ns:]).reshape(2, 3, 8, 8) for p in parts])
        assert np.array_equal(y, y_ref) and np.array_equal(s, s_ref)


def test_single_process_identity():
    import bench
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert bench.rank_layer(0) == 0
