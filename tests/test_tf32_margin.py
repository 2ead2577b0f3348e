"""The TF32 path's error margin, and where its error comes from.

CPU: the error model of tests/tf32_error_model.py (the chunked forward in
float64 with each rounding source of the kernels switchable) against the
oracle, on a single-layer-like problem. It pins the model (exact mode equals the
oracle; TF32 rounding of a known value) and shows that the operand rounding to
TF32 is the error: the float32 in-chunk cumulative sum, exponentials and state
pass add 1e-6 or less. The tensor core drops the 13 low bits of an fp32 operand
(its measured error, 1.47e-3 on y at the single-layer shape, matches truncation,
not rounding to nearest), so the kernels round the operands they write
themselves (P, x, dec o B, C', and the staged path's windows and transposes) to
nearest; the model gives the error of that mix, about 8e-4 on y, 3e-4 on the
state.

GPU: ten seeds at the single-layer shape and at a long-memory shape (1024
chunks, slow decay), every result within 1e-3 of the oracle on y and the final
state (half the 2e-3 tolerance; the largest is printed in the session summary).
"""
import numpy as np
import pytest

from oracle import naive_scan_inputs
from state_space_sequence_complex_gb300 import inputs
from tests.tf32_error_model import chunked_forward, round_tf32

rel = lambda a, b: float(np.linalg.norm(a - b) / np.linalg.norm(b))


def test_tf32_rounding_of_known_values():
    one_plus = np.float32(1.0) + np.float32(2.0 ** -11)  # half an ulp of TF32 at 1
    assert round_tf32(np.array([one_plus]), "rz")[0] == 1.0
    assert round_tf32(np.array([one_plus]), "rn")[0] == 1.0  # tie to even
    above = np.float32(1.0) + np.float32(2.0 ** -11) + np.float32(2.0 ** -20)
    assert round_tf32(np.array([above]), "rn")[0] == 1.0 + 2.0 ** -10
    assert round_tf32(np.array([-above]), "rz")[0] == -1.0
    assert round_tf32(np.array([np.float32(3.0)]), "rn")[0] == 3.0
    assert round_tf32(np.array([one_plus]), "rna")[0] == 1.0 + 2.0 ** -10  # tie away from zero
    assert round_tf32(np.array([-one_plus]), "rna")[0] == -(1.0 + 2.0 ** -10)


@pytest.fixture(scope="module")
def layer_like():
    inp = inputs.custom(1, 512, 4, 64, 64, seed=1)
    return inp, inp.complex(), naive_scan_inputs(inp)


def _err(layer_like, **kw):
    _, c, (y_ref, s_ref) = layer_like
    y, s = chunked_forward(c["x"], c["A"], c["B"], c["C"], c["dt"], 64, **kw)
    return rel(y, y_ref), rel(s, s_ref)


def test_model_exact_mode_is_the_oracle(layer_like):
    ey, es = _err(layer_like)
    assert ey < 1e-12 and es < 1e-12


def test_float32_sources_are_negligible(layer_like):
    for kw in (dict(acs32=True), dict(exp32=True), dict(state32=True)):
        ey, es = _err(layer_like, **kw)
        assert ey < 1e-5 and es < 1e-5, kw


def test_operand_rounding_dominates_and_the_kernels_mix_is_below_1e3(layer_like):
    rz = _err(layer_like, operands="rz")
    rn = _err(layer_like, operands="rn")
    assert rn[0] < rz[0] / 2 and rn[1] < rz[1] / 2
    # truncation alone: the error the kernels had before rounding their operands
    assert 1e-3 < rz[0] < 2e-3
    # the kernels: P, x, dec o B and C' rounded to nearest; C, B (read by the MMA as loaded)
    # and S_in (kept in float32 for the state pass) truncated by the tensor core
    mix = _err(layer_like, operands="rna", loaded="rz", state_op="rz", acs32=True, exp32=True, state32=True)
    assert mix[0] < 1e-3 and mix[1] < 1e-3


@pytest.mark.gpu
@pytest.mark.parametrize("shape", ["single_layer", "long_memory"])
def test_tf32_error_across_seeds(shape):
    from state_space_sequence_complex_gb300 import build, ssdc
    from tests.gpu_util import assert_close, run_library
    build.build()
    ssdc.load()
    worst = [0.0, 0.0]
    for seed in range(10):
        if shape == "single_layer":
            inp = inputs.custom(2, 2048, 16, 64, 64, seed=7000 + seed)
        else:  # the long-memory distributions: slow decay, small steps, 1024 chunks
            inp = inputs.custom(1, 65536, 2, 64, 64, seed=7100 + seed, re_lo=-0.1, re_hi=-0.01,
                                dt_mean=-2.0, dt_std=0.5)
        y, s, _ = run_library(inp, 64, "tf32")
        ey, es = assert_close(y, s, *naive_scan_inputs(inp), "tf32", f"{shape} seed {seed}")
        worst = [max(worst[0], ey), max(worst[1], es)]
    assert worst[0] <= 1e-3 and worst[1] <= 1e-3, worst
