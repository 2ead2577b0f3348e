"""The bench's multi-rank logic on CPU with two gloo ranks: each rank gets its
own independently seeded batch, and timings are reduced by max over ranks."""
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


def test_single_process_identity():
    import bench
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert bench.rank_layer(0) == 0
