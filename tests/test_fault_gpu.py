"""Failure detection without a GPU fault: a test hook makes one chunk of the
fused kernel skip sending its state; the receiving CTA's wait gives up after
its 2 s limit and the call reports SSDC_ERR_TIMEOUT through the workspace
status. The context stays usable: the next call is correct."""
import pytest

from oracle import naive_scan_inputs
from state_space_sequence_complex_gb300 import inputs, ssdc
from tests.gpu_util import assert_close, run_library, to_device

pytestmark = pytest.mark.gpu

ORDER = ["x_re", "x_im", "A_re", "A_im", "B_re", "B_im", "C_re", "C_im", "dt"]


@pytest.fixture(scope="module", autouse=True)
def built():
    from state_space_sequence_complex_gb300 import build
    build.build()
    ssdc.load()


def test_dropped_state_times_out_then_recovers(lib_option):
    import torch
    lib_option(ssdc.OPT_FUSED_CLUSTER, 2)
    inp = inputs.custom(1, 128, 1, 64, 64, seed=5)  # two chunks on a 2-CTA cluster
    dev = to_device(inp)
    f = ssdc.Forward(*inp.dims, 64, "tf32")
    lib_option(ssdc.OPT_TEST_DROP_STATE_CHUNK, 0)
    f(*[dev[k] for k in ORDER])
    torch.cuda.synchronize()
    assert f.status() == ssdc.SSDC_ERR_TIMEOUT
    lib_option(ssdc.OPT_TEST_DROP_STATE_CHUNK, -1)
    y, s, _ = run_library(inp, 64, "tf32", dev=dev, forward=f)
    assert_close(y, s, *naive_scan_inputs(inp), "tf32", "after a timed-out call")
