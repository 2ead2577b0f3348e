"""Repeat-determinism of the tensor-core kernels, as a race detector.

Every kernel here hands tiles, accumulators and states between warps, CTAs
and the tensor cores through mbarriers, named barriers and (in the cluster
kernel) distributed shared memory; none of its sums depends on arrival order.
So a missing wait or release (a warp reading a tile before it is written, a
TMA load overwriting a tile still being read, a state hop read early) shows
as a run-to-run difference, while a correct kernel returns the same bits
every time. Each case runs once, then again many times with unrelated
launches of varying size in between (which shift the timing of the CTAs
against each other), and every output must equal the first run's bit for
bit. Cases: the cluster kernel at 1, 2, 4 and 8 CTAs per sequence (with and
without an initial state), the tensor-memory kernel at every chunk size, its
bfloat16-input and fused head-mixer instances, the scan followed by the
separate head mixer, the final state alone
(ssd_complex_final_state), the staged TF32 path, and the TF32 backward
(whose chunk kernels walk several chunks a CTA, loading the next chunk's
tiles as the current one frees them).
"""
import numpy as np
import pytest
import torch

from state_space_sequence_complex_gb300 import inputs, ssdc
from tests.gpu_util import to_device

pytestmark = pytest.mark.gpu

ORDER = ["x_re", "x_im", "A_re", "A_im", "B_re", "B_im", "C_re", "C_im", "dt"]
REPEATS = 12


@pytest.fixture(scope="module", autouse=True)
def built():
    from state_space_sequence_complex_gb300 import build
    build.build()
    ssdc.load()


def repeat_identical(call, status, expect_path):
    """call() -> tuple of device tensors (the library's own output buffers).
    Runs it REPEATS + 1 times, perturbing the timing in between, and checks
    that every run returns the first run's bits."""
    first = [t.clone() for t in call()]
    torch.cuda.synchronize()
    assert status() == ssdc.SSDC_OK, ssdc.strerror(status())
    if expect_path is not None:  # (the backward records no path)
        assert ssdc.last_path() == expect_path, ssdc.last_path()
    rng = np.random.default_rng(11)
    pad = torch.empty(1 << 24, dtype=torch.float32, device="cuda")
    for r in range(REPEATS):
        pad[: int(rng.integers(1, 1 << 24))].fill_(float(r))  # an unrelated launch of varying size
        out = call()
        torch.cuda.synchronize()
        assert status() == ssdc.SSDC_OK, ssdc.strerror(status())
        for k, (a, b) in enumerate(zip(first, out)):
            if not torch.equal(a, b):
                diff = (a - b).abs().max().item()
                raise AssertionError(f"run {r + 1}: output {k} differs from the first run (max |diff| {diff:.3e})")


def forward_call(inp, Q, precision, s0=False, bf16=False):
    t = to_device(inp)
    if bf16:
        for k in ("x_re", "x_im", "B_re", "B_im", "C_re", "C_im"):
            t[k] = t[k].to(torch.bfloat16)
    f = ssdc.Forward(*inp.dims, Q, precision, bf16_inputs=bf16) if bf16 else ssdc.Forward(*inp.dims, Q, precision)
    kw = {}
    if s0:
        Bn, T, H, N, D = inp.dims
        g = torch.Generator(device="cuda").manual_seed(5)
        kw = dict(s0_re=torch.randn(Bn, H, N, D, device="cuda", generator=g) * 4,
                  s0_im=torch.randn(Bn, H, N, D, device="cuda", generator=g) * 4)
    return (lambda: f(*[t[k] for k in ORDER], **kw)), f.status


@pytest.mark.parametrize("cl", [1, 2, 4, 8])
def test_cluster_kernel_repeats_bit_for_bit(lib_option, cl):
    lib_option(ssdc.OPT_FUSED_KERNEL, 1)
    lib_option(ssdc.OPT_FUSED_CLUSTER, cl)
    inp = inputs.generate(inputs.LAYER)  # the single-layer shape, 32 sequences of 32 chunks
    call, status = forward_call(inp, 64, "tf32")
    repeat_identical(call, status, "fused_cluster")


def test_cluster_kernel_initial_state_repeats_bit_for_bit(lib_option):
    lib_option(ssdc.OPT_FUSED_KERNEL, 1)
    lib_option(ssdc.OPT_FUSED_CLUSTER, 4)
    inp = inputs.custom(3, 64 * 9 + 13, 8, 64, 64, seed=31)
    call, status = forward_call(inp, 64, "tf32", s0=True)
    repeat_identical(call, status, "fused_cluster")


@pytest.mark.parametrize("Q", [16, 32, 64, 128, 256])
def test_tmem_kernel_repeats_bit_for_bit(lib_option, Q):
    lib_option(ssdc.OPT_FUSED_KERNEL, 2)
    inp = inputs.custom(20, 1000, 16, 64, 64, seed=40 + Q)  # 320 sequences: two or three per CTA, ragged tail
    call, status = forward_call(inp, Q, "tf32", s0=(Q == 64))
    repeat_identical(call, status, "fused_tmem")


@pytest.mark.parametrize("Q", [64, 128])
def test_bf16_inputs_repeat_bit_for_bit(Q):
    inp = inputs.custom(20, 1000, 16, 64, 64, seed=50 + Q)
    call, status = forward_call(inp, Q, "tf32", bf16=True)
    repeat_identical(call, status, "fused_tmem")


@pytest.mark.parametrize("fused", [0, 1], ids=["separate_mixer", "fused_mixer"])
def test_mixer_repeats_bit_for_bit(fused, lib_option):
    lib_option(ssdc.OPT_MIMO_FUSED, fused)
    inp = inputs.custom(20, 1000, 16, 64, 64, seed=60)
    t = to_device(inp)
    W = torch.from_numpy((np.eye(16) + 0.3 * np.random.default_rng(61).standard_normal((16, 16)))
                         .astype(np.float32)).cuda()
    f = ssdc.MimoForward(*inp.dims, 64)
    repeat_identical(lambda: f(*[t[k] for k in ORDER], W), f.status, "fused_tmem")


def test_staged_tf32_repeats_bit_for_bit():
    inp = inputs.custom(4, 1000, 16, 64, 64, seed=70)
    call, status = forward_call(inp, 128, "tf32_staged")
    repeat_identical(call, status, "staged_tf32")


@pytest.mark.parametrize("Q", [64, 256])
def test_final_state_alone_repeats_bit_for_bit(Q):
    inp = inputs.custom(20, 1000, 16, 64, 64, seed=80 + Q)
    t = to_device(inp)
    f = ssdc.FinalState(*inp.dims, Q, "tf32")
    repeat_identical(lambda: f(*[t[k] for k in ("x_re", "x_im", "A_re", "A_im", "B_re", "B_im", "dt")]), f.status,
                     "state_tmem")


@pytest.mark.parametrize("Q,real", [(64, False), (32, True)])
def test_tf32_backward_repeats_bit_for_bit(Q, real):
    Bn, T, H, D, N = 4, 1000, 16, 64, 64
    inp = inputs.custom(Bn, T, H, D, N, seed=90 + Q)
    og = inputs.output_grads(Bn, T, H, D, N, seed=91 + Q)
    t = to_device(inp)
    if real:  # a real x and a loss of Re(y): the kernels zero the imaginary planes again each chunk
        t["x_im"] = None
    cu = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    dy_re, dy_im = cu(og.dy_re), None if real else cu(og.dy_im)
    dfs_re, dfs_im = cu(og.dfs_re), cu(og.dfs_im)
    b = ssdc.Backward(Bn, T, H, N, D, Q, precision="tf32")
    keys = ["dx_re", "dA_re", "dA_im", "dB_re", "dB_im", "dC_re", "dC_im", "ddt"] + ([] if real else ["dx_im"])

    def call():
        g = b(*[t[k] for k in ORDER], dy_re, dy_im, dfs_re, dfs_im)
        return tuple(g[k] for k in keys)

    repeat_identical(call, lambda: ssdc.ssd_complex_status(b.workspace), None)
