"""GPU parity: the library (through the C ABI) against the CPU oracle, element
by element, relative Frobenius error on y (B,T,H,D) and the final state
(B,H,N,D): <= 1e-5 on the exact fp32 path, <= 2e-3 on the TF32 path."""
import numpy as np
import pytest

from oracle import naive_scan_inputs
from state_space_sequence_complex_gb300 import inputs, ssdc
from tests.gpu_util import TOL, assert_close, rel_fro, run_library, to_device

pytestmark = pytest.mark.gpu

PRECISIONS = ["fp32", "tf32"]


@pytest.fixture(scope="session", autouse=True)
def built():
    from state_space_sequence_complex_gb300 import build
    build.build()
    ssdc.load()


def supported(inp, Q, precision):
    Bn, T, H, N, D = inp.dims
    return ssdc.ssd_complex_fwd_supported(ssdc.dims(Bn, T, H, N, D, precision), Q) == 0


def check(inp, Q, precision, what="", ref=None):
    if not supported(inp, Q, precision):
        pytest.skip(f"{precision} does not support Q={Q}, dims {inp.dims}")
    y_ref, s_ref = ref if ref is not None else naive_scan_inputs(inp)
    y, s, _ = run_library(inp, Q, precision)
    return assert_close(y, s, y_ref, s_ref, precision, what)


@pytest.mark.parametrize("precision", PRECISIONS)
@pytest.mark.parametrize("w", [inputs.TINY, inputs.TINY_DT0], ids=["dt_normal", "dt_zero"])
def test_tiny_workload(w, precision):
    check(inputs.generate(w), w.Q, precision, w.name)


@pytest.mark.parametrize("precision", PRECISIONS)
@pytest.mark.parametrize("T,Q", [(64, 64), (100, 64), (10, 64), (1, 64), (257, 32), (300, 128),
                                 (511, 256), (1000, 64), (64, 16), (90, 16)])
def test_uneven_and_edge_lengths(T, Q, precision):
    inp = inputs.custom(2, T, 3, 64, 64, seed=1000 + T + Q)
    check(inp, Q, precision, f"T={T} Q={Q}")


@pytest.mark.parametrize("precision", PRECISIONS)
@pytest.mark.parametrize("N,D", [(8, 8), (16, 64), (64, 8), (32, 24), (56, 40)])
def test_state_and_head_sizes(N, D, precision):
    inp = inputs.custom(2, 200, 3, D, N, seed=N * 100 + D)
    check(inp, 64, precision, f"N={N} D={D}")


# The fused kernel with the state in tensor memory, forced: every chunk size it takes
# (chunks of 128 and 256 tokens as 3 and 10 blocks of 64 x 64), feature sizes below the
# tile (zero columns), ragged tails (inside the last block, and whole blocks past T),
# T < Q, T = Q.
@pytest.mark.parametrize("N,D,Q,T", [(8, 8, 16, 128), (8, 8, 16, 90), (16, 64, 32, 257), (64, 8, 64, 200),
                                     (32, 24, 16, 333), (56, 40, 32, 1000), (64, 64, 16, 300), (64, 64, 32, 1000),
                                     (64, 64, 64, 64 * 9 + 13), (24, 48, 32, 20), (64, 64, 64, 64), (8, 16, 16, 1),
                                     (64, 64, 128, 300), (64, 64, 128, 3 * 128), (16, 40, 128, 1000),
                                     (8, 8, 128, 129), (64, 64, 256, 511), (64, 64, 256, 256), (32, 64, 256, 700),
                                     (64, 64, 256, 70), (48, 16, 256, 1030)])
def test_tensor_memory_kernel(N, D, Q, T, lib_option):
    lib_option(ssdc.OPT_FUSED_KERNEL, 2)
    inp = inputs.custom(2, T, 3, D, N, seed=5000 + N + D + Q + T)
    check(inp, Q, "tf32", f"tensor-memory kernel N={N} D={D} Q={Q} T={T}")


@pytest.mark.parametrize("Q", [32, 64, 128, 256])
def test_tensor_memory_kernel_several_sequences_per_cta(Q, lib_option):
    # 160 sequences on at most 152 CTAs: some CTAs walk two sequences
    lib_option(ssdc.OPT_FUSED_KERNEL, 2)
    inp = inputs.custom(20, 200, 8, 64, 64, seed=5100 + Q)
    check(inp, Q, "tf32", f"160 sequences Q={Q}")


def test_both_fused_kernels_on_one_problem(lib_option):
    # the same inputs through the cluster kernel (forced 2-CTA clusters) and the
    # tensor-memory kernel: each against the oracle
    inp = inputs.custom(3, 64 * 7 + 5, 5, 64, 64, seed=5200)
    ref = naive_scan_inputs(inp)
    out = {}
    for kernel in (1, 2):
        lib_option(ssdc.OPT_FUSED_KERNEL, kernel)
        if kernel == 1:
            lib_option(ssdc.OPT_FUSED_CLUSTER, 2)
        y, s, _ = run_library(inp, 64, "tf32")
        assert_close(y, s, *ref, "tf32", f"fused kernel {kernel}")
        out[kernel] = (y, s)
    assert rel_fro(out[1][0], out[2][0]) <= TOL["tf32"]


@pytest.mark.parametrize("precision", PRECISIONS)
def test_chunk_size_invariance(precision):
    # same inputs for every Q, all against one oracle result (landing page: chunked == naive)
    inp = inputs.custom(2, 1024, 4, 64, 64, seed=77)
    ref = naive_scan_inputs(inp)
    for Q in (16, 32, 64, 128, 256):
        if supported(inp, Q, precision):
            check(inp, Q, precision, f"Q={Q}", ref=ref)


@pytest.mark.parametrize("precision", PRECISIONS)
def test_production_layer(precision):
    w = inputs.LAYER
    check(inputs.generate(w), w.Q, precision, w.name)


@pytest.mark.parametrize("precision", PRECISIONS)
def test_positive_real_part_short(precision):
    # the pages' Skill-2 example draws A = randn - 1, so Re(A) > 0 (growth) is allowed
    inp = inputs.custom(2, 64, 2, 64, 64, seed=5, re_lo=-1.0, re_hi=0.3)
    check(inp, 64 if precision == "tf32" else 16, precision, "Re(A) > 0")


def test_fp32_is_deterministic():
    inp = inputs.custom(2, 500, 4, 64, 64, seed=3)
    dev = to_device(inp)
    y1, s1, f = run_library(inp, 64, "fp32", dev=dev)
    y2, s2, _ = run_library(inp, 64, "fp32", dev=dev, forward=f)
    assert np.array_equal(y1, y2) and np.array_equal(s1, s2)


def test_launch_count_and_reuse():
    inp = inputs.custom(1, 256, 2, 64, 64, seed=4)
    dev = to_device(inp)
    _, _, f = run_library(inp, 64, "fp32", dev=dev)
    assert ssdc.last_launch_count() == 3
    ref = naive_scan_inputs(inp)
    # a second call on the same workspace gives the same answer
    y, s, _ = run_library(inp, 64, "fp32", dev=dev, forward=f)
    assert_close(y, s, *ref, "fp32")


@pytest.mark.parametrize("T,Q", [(64, 64), (1000, 64), (300, 128), (511, 256), (100, 64), (257, 32), (32, 32),
                                 (31, 32), (1000, 32)])
def test_staged_tf32_path(T, Q):
    inp = inputs.custom(2, T, 3, 64, 64, seed=2000 + T + Q)
    check(inp, Q, "tf32_staged", f"staged T={T} Q={Q}")


@pytest.mark.parametrize("cluster", [1, 2, 4, 8])
def test_fused_cluster_sizes(cluster, lib_option):
    # several sequences per cluster, a partial last chunk, more chunks than CTAs
    lib_option(ssdc.OPT_FUSED_CLUSTER, cluster)
    inp = inputs.custom(2, 64 * 9 + 13, 3, 64, 64, seed=3000 + cluster)
    check(inp, 64, "tf32", f"fused cluster {cluster}")


def test_fused_fewer_chunks_than_cluster(lib_option):
    lib_option(ssdc.OPT_FUSED_CLUSTER, 8)
    inp = inputs.custom(1, 130, 2, 64, 64, seed=31)   # 3 chunks on an 8-CTA cluster
    check(inp, 64, "tf32", "3 chunks, cluster 8")


def test_fused_single_launch_and_small_workspace():
    d = ssdc.dims(2, 2048, 16, 64, 64, "tf32")
    assert ssdc.ssd_complex_fwd_workspace_bytes(d, 64) == 256
    inp = inputs.custom(1, 256, 2, 64, 64, seed=8)
    _, _, f = run_library(inp, 64, "tf32")
    assert ssdc.last_launch_count() == 1


def _planes_in_order(t, name, imag_first):
    """Both planes of one tensor in one allocation, in the given address order."""
    import torch
    re, im = t[name + "_re"], t[name + "_im"]
    buf = torch.empty((2,) + tuple(re.shape), dtype=re.dtype, device=re.device)
    first, second = (im, re) if imag_first else (re, im)
    buf[0].copy_(first)
    buf[1].copy_(second)
    t[name + "_re"], t[name + "_im"] = (buf[1], buf[0]) if imag_first else (buf[0], buf[1])


@pytest.mark.parametrize("kernel", [1, 2])
@pytest.mark.parametrize("plane_maps", ["1", "0"])
@pytest.mark.parametrize("order", ["re_first", "im_first", "mixed"])
def test_fused_tensor_map_paths(order, plane_maps, kernel, lib_option):
    # T a multiple of 8 (the interleaved C map applies) with a partial last chunk; each
    # tensor's planes either in one map (in either address order) or in one map per plane;
    # the cluster kernel (2-CTA clusters) and the tensor-memory kernel
    lib_option(ssdc.OPT_FUSED_KERNEL, kernel)
    if kernel == 1:
        lib_option(ssdc.OPT_FUSED_CLUSTER, 2)
    lib_option(ssdc.OPT_FUSED_PLANE_MAPS, int(plane_maps))
    inp = inputs.custom(2, 64 * 5 + 24, 3, 64, 64, seed=3100)
    y_ref, s_ref = naive_scan_inputs(inp)
    t = to_device(inp)
    flips = {"re_first": (False, False, False), "im_first": (True, True, True), "mixed": (True, False, True)}[order]
    for name, flip in zip(["x", "B", "C"], flips):
        _planes_in_order(t, name, flip)
    y, s, _ = run_library(inp, 64, "tf32", dev=t)
    assert_close(y, s, y_ref, s_ref, "tf32", f"planes {order}, plane maps {plane_maps}")


@pytest.mark.parametrize("Q", [128, 256])
@pytest.mark.parametrize("plane_maps", ["1", "0"])
def test_tensor_memory_kernel_map_paths_long_chunks(Q, plane_maps, lib_option):
    # chunks of several 64-token blocks through each tensor-map form (T a multiple of 8:
    # the interleaved C map applies), planes in mixed address order
    lib_option(ssdc.OPT_FUSED_PLANE_MAPS, int(plane_maps))
    inp = inputs.custom(2, 2 * Q + 72, 3, 64, 64, seed=3200 + Q)
    y_ref, s_ref = naive_scan_inputs(inp)
    t = to_device(inp)
    for name, flip in zip(["x", "B", "C"], (True, False, True)):
        _planes_in_order(t, name, flip)
    y, s, _ = run_library(inp, Q, "tf32", dev=t)
    assert ssdc.last_path() == "fused_tmem"
    assert_close(y, s, y_ref, s_ref, "tf32", f"Q={Q}, plane maps {plane_maps}")
