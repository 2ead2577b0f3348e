"""The host-buffer entry point (ssd_complex_fwd_host): inputs and outputs in
host memory, the library copying pieces of the problem in and out around the
scan. Checked against the oracle on small cases that exercise each way of
cutting the problem (segments of the sequence carried by the initial-state
path for a small batch, groups of batch rows for a large one, a partial last
segment or group), with pinned and with pageable host buffers, and against the
device entry point at the single-layer size and with more pieces than device
slots."""
import numpy as np
import pytest
import torch

from oracle import naive_scan_inputs
from state_space_sequence_complex_gb300 import inputs, ssdc
from tests.gpu_util import TOL, assert_close, rel_fro, run_library

pytestmark = pytest.mark.gpu

ORDER = ["x_re", "x_im", "A_re", "A_im", "B_re", "B_im", "C_re", "C_im", "dt"]


@pytest.fixture(scope="module", autouse=True)
def built():
    from state_space_sequence_complex_gb300 import build
    build.build()
    ssdc.load()


def host_inputs(inp, pinned):
    out = {}
    for k, v in inp.arrays().items():
        t = torch.from_numpy(np.ascontiguousarray(v))
        out[k] = t.pin_memory() if pinned else t.clone()
    return out


def run_host(inp, Q, precision, pinned=True):
    h = host_inputs(inp, pinned)
    f = ssdc.HostForward(*inp.dims, Q, precision)
    y_re, y_im, fs_re, fs_im = f(*[h[k] for k in ORDER])
    y = y_re.double().numpy() + 1j * y_im.double().numpy()
    s = fs_re.double().numpy() + 1j * fs_im.double().numpy()
    return y, s


# (B, T, H, D, N, Q, precision). A batch of fewer than 4 rows goes as up to 4
# segments of the sequence (a multiple of Q tokens each, the last partial), each
# started from the previous one's final state; 4 rows or more go as up to 4 row
# groups (B = 5 and 9 give a smaller last group).
CASES = [
    (1, 200, 2, 16, 16, 32, "fp32"),
    (1, 100, 3, 8, 8, 16, "fp32"),
    (2, 130, 6, 8, 24, 16, "fp32"),
    (5, 96, 3, 16, 8, 64, "fp32"),
    (9, 64, 2, 8, 8, 16, "fp32"),
    (1, 256, 4, 64, 64, 64, "tf32"),
    (2, 320, 4, 64, 64, 64, "tf32"),
    (5, 128, 2, 64, 64, 64, "tf32"),
    (2, 200, 2, 64, 64, 128, "tf32"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}T{}H{}D{}N{}Q{}-{}".format(*c))
def test_host_entry_matches_oracle(case):
    Bn, T, H, D, N, Q, precision = case
    inp = inputs.custom(Bn, T, H, D, N, seed=300 + Bn * 7 + H)
    y_ref, s_ref = naive_scan_inputs(inp)
    y, s = run_host(inp, Q, precision)
    assert_close(y, s, y_ref, s_ref, precision, "host buffers")
    if precision == "fp32":
        # each (b, h) sequence runs the same exact-fp32 arithmetic whatever piece it is in:
        # segments start at chunk boundaries and carry the state the whole scan would
        yd, sd, _ = run_library(inp, Q, precision)
        assert np.array_equal(y, yd) and np.array_equal(s, sd)


def test_host_entry_pageable_buffers():
    inp = inputs.custom(3, 160, 4, 16, 16, seed=331)
    y_ref, s_ref = naive_scan_inputs(inp)
    y, s = run_host(inp, 32, "fp32", pinned=False)
    assert_close(y, s, y_ref, s_ref, "fp32", "pageable host buffers")


def test_host_entry_single_layer_matches_device_entry():
    inp = inputs.generate(inputs.LAYER)
    y, s = run_host(inp, 64, "tf32")
    assert ssdc.last_launch_count() == 4  # 4 segments of 512 tokens, one fused launch each
    yd, sd, _ = run_library(inp, 64, "tf32")
    assert rel_fro(y, yd) <= 1e-6 and rel_fro(s, sd) <= 1e-6


@pytest.mark.parametrize("precision", ["fp32", "tf32"])
def test_host_entry_more_pieces_than_slots(precision):
    # 538 MB of inputs and outputs: 8 pieces of 1 batch row through the 2 device slots
    inp = inputs.custom(8, 2048, 16, 64, 64, seed=351)
    y, s = run_host(inp, 64, precision)
    assert ssdc.last_launch_count() == 8 * (1 if precision == "tf32" else 3)
    yd, sd, _ = run_library(inp, 64, precision)
    if precision == "fp32":
        assert np.array_equal(y, yd) and np.array_equal(s, sd)
    else:
        assert rel_fro(y, yd) <= 1e-6 and rel_fro(s, sd) <= 1e-6


def test_host_entry_repeated_calls_reuse_scratch():
    a = inputs.custom(4, 128, 2, 64, 64, seed=341)
    b = inputs.custom(4, 128, 2, 64, 64, seed=342)
    f = ssdc.HostForward(*a.dims, 64, "tf32")
    for inp in (a, b, a):
        h = host_inputs(inp, True)
        y_re, y_im, fs_re, fs_im = f(*[h[k] for k in ORDER])
        y_ref, s_ref = naive_scan_inputs(inp)
        y = y_re.double().numpy() + 1j * y_im.double().numpy()
        s = fs_re.double().numpy() + 1j * fs_im.double().numpy()
        assert_close(y, s, y_ref, s_ref, "tf32", "repeated host call")
