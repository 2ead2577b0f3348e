"""GPU parity at the full benchmark sizes, in the launch configuration the
bench times (one Forward object, workspace preallocated)."""
import numpy as np
import pytest

from oracle import naive_scan
from state_space_sequence_complex_gb300 import inputs, ssdc
from tests.gpu_util import assert_close, run_library, to_device

pytestmark = pytest.mark.gpu

PRECISIONS = ["fp32", "tf32"]


def _supported(inp, Q, precision):
    Bn, T, H, N, D = inp.dims
    return ssdc.ssd_complex_fwd_supported(ssdc.dims(Bn, T, H, N, D, precision), Q) == 0


def _oracle(inp, **kw):
    a = inp.arrays()
    return naive_scan(a["x_re"], a["x_im"], a["A_re"], a["A_im"], a["B_re"], a["B_im"],
                      a["C_re"], a["C_im"], a["dt"], **kw)


@pytest.fixture(scope="module")
def long_case():
    inp = inputs.generate(inputs.LONG)
    return inp, _oracle(inp)


@pytest.mark.parametrize("precision", PRECISIONS)
def test_long_memory_full(long_case, precision):
    inp, (y_ref, s_ref) = long_case
    if not _supported(inp, 64, precision):
        pytest.skip("unsupported")
    y, s, _ = run_library(inp, 64, precision)
    assert_close(y, s, y_ref, s_ref, precision, inputs.LONG.name)


@pytest.fixture(scope="module")
def qsweep_case():
    inp = inputs.generate(inputs.QSWEEP)
    # oracle y on the 512-token prefix, state over the full length
    return inp, _oracle(inp, t_y=512)


@pytest.mark.parametrize("precision", PRECISIONS)
@pytest.mark.parametrize("Q", [32, 64, 128, 256])
def test_chunk_sweep_prefix_and_state(qsweep_case, Q, precision):
    inp, (y_ref, s_ref) = qsweep_case
    if not _supported(inp, Q, precision):
        pytest.skip("unsupported")
    y, s, _ = run_library(inp, Q, precision)
    assert_close(y[:, :512], s, y_ref[:, :512], s_ref, precision, f"sweep Q={Q}")


@pytest.mark.parametrize("precision", PRECISIONS)
def test_training_batch_28_layers_sampled(precision):
    # every layer runs at full size on the GPU; the oracle checks batch rows 0 and 15
    w = inputs.TRAIN28
    f = None
    for layer in range(w.layers):
        inp = inputs.generate(w, layer=layer)
        dev = to_device(inp)
        y, s, f = run_library(inp, w.Q, precision, dev=dev, forward=f)
        rows = [0, w.B - 1]
        sub = inputs.Inputs(**{k: (v[rows] if v.ndim > 1 else v) for k, v in inp.arrays().items()})
        y_ref, s_ref = _oracle(sub)
        assert_close(y[rows], s[rows], y_ref, s_ref, precision, f"layer {layer}")
        del dev
