"""The data-parallel backward on CPU with two gloo ranks: each rank holds one
batch row of a problem and its gradients; the all-reduce of dA over the ranks
(bench.reduce_param_grads) gives the whole batch's dA, and every other
gradient of a row is the whole batch's gradient of that row. Gradients come
from the gradient oracle (no GPU)."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

SHAPE = dict(Bn=2, T=150, H=3, D=4, N=5)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem():
    from state_space_sequence_complex_gb300 import inputs
    Bn, T, H, D, N = (SHAPE[k] for k in ("Bn", "T", "H", "D", "N"))
    inp = inputs.custom(Bn, T, H, D, N, seed=901)
    og = inputs.output_grads(Bn, T, H, D, N, seed=902)
    return inp, og


def _rows(inp, og, b):
    from state_space_sequence_complex_gb300 import inputs
    a = {k: (v if v.ndim == 1 else np.ascontiguousarray(v[b:b + 1])) for k, v in inp.arrays().items()}
    g = inputs.OutputGrads(og.dy_re[b:b + 1], og.dy_im[b:b + 1], og.dfs_re[b:b + 1], og.dfs_im[b:b + 1])
    return inputs.Inputs(**a), g


def _worker(rank, world, port, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    from oracle import naive_grad_inputs
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        inp, og = _problem()
        mine, g = _rows(inp, og, rank)
        grads = naive_grad_inputs(mine, g.dy_re + 1j * g.dy_im, g.dfs_re + 1j * g.dfs_im, threads=1)
        dA_re = torch.tensor(grads["dA"].real)
        dA_im = torch.tensor(grads["dA"].imag)
        bench.reduce_param_grads(dA_re, dA_im)
        out[rank] = (dA_re.numpy() + 1j * dA_im.numpy(), grads["dx"], grads["ddt"])
    finally:
        dist.destroy_process_group()


def test_data_parallel_backward_two_gloo_ranks():
    from oracle import naive_grad_inputs
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    inp, og = _problem()
    full = naive_grad_inputs(inp, og.dy_re + 1j * og.dy_im, og.dfs_re + 1j * og.dfs_im, threads=1)
    for rank in range(2):
        dA, dx, ddt = out[rank]
        # the sum of two per-row shares, in either order, is the whole batch's dA
        assert np.array_equal(dA, full["dA"])
        assert np.array_equal(dx, full["dx"][rank:rank + 1])
        assert np.array_equal(ddt, full["ddt"][rank:rank + 1])


def test_reduce_is_identity_on_one_process():
    import bench
    a, b = torch.tensor([1.0, 2.0]), torch.tensor([3.0, 4.0])
    bench.reduce_param_grads(a, b)
    assert a.tolist() == [1.0, 2.0] and b.tolist() == [3.0, 4.0]
