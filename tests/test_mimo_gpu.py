"""The forward pass with the MIMO head mixer (NEXT-3: ssd_complex_fwd_mimo),
on both of its paths: the scan followed by the separate in-place mixer kernel
(the default, two launches) and the mixer fused into the scan's epilogue
(SSDC_OPT_MIMO_FUSED = 1, one launch). The mixed Re(y) against the oracle's scan followed by
the oracle's head mixer, at the TF32 tolerance (relative Frobenius error 2e-3
on the output and the final state). With the identity matrix (the pages'
initialisation) the output is the plain forward's Re(y), bit for bit. Cases:
the single-layer shape, Q = 16 / 32 / 64, ragged tails, H below 16, N and D
below 64, several sequences per CTA, an initial state, a real x."""
import numpy as np
import pytest
import torch

from oracle import head_mix, naive_scan, naive_scan_inputs
from state_space_sequence_complex_gb300 import inputs, ssdc
from tests.gpu_util import assert_close, to_device

pytestmark = pytest.mark.gpu

ORDER = ["x_re", "x_im", "A_re", "A_im", "B_re", "B_im", "C_re", "C_im", "dt"]


@pytest.fixture(scope="module", autouse=True)
def built():
    from state_space_sequence_complex_gb300 import build
    build.build()
    ssdc.load()


@pytest.fixture(params=["separate", "fused"], autouse=True)
def mimo_path(request, lib_option):
    if request.param == "fused":
        lib_option(ssdc.OPT_MIMO_FUSED, 1)
    return request.param


def mixing_matrix(H, seed):
    # identity plus a cross-head part of the size training would give it
    rng = np.random.default_rng(seed)
    return (np.eye(H) + 0.3 * rng.standard_normal((H, H))).astype(np.float32)


def run_mimo(inp, Q, W, s0=None, real_x=False, launches=None):
    t = to_device(inp)
    if real_x:
        t["x_im"] = None
    f = ssdc.MimoForward(*inp.dims, Q)
    kw = {}
    if s0 is not None:
        kw = dict(s0_re=torch.from_numpy(np.ascontiguousarray(s0.real, dtype=np.float32)).cuda(),
                  s0_im=torch.from_numpy(np.ascontiguousarray(s0.imag, dtype=np.float32)).cuda())
    out, fs_re, fs_im = f(*[t[k] for k in ORDER], torch.from_numpy(W).cuda(), **kw)
    torch.cuda.synchronize()
    assert f.status() == ssdc.SSDC_OK
    # the fused epilogue runs on the tensor-memory kernel; the separate mixer follows whichever
    # fused kernel the library picks for the scan
    assert ssdc.last_path() in (("fused_tmem",) if launches == 1 else ("fused_tmem", "fused_cluster"))
    if launches is not None:
        assert ssdc.last_launch_count() == launches
    return out.double().cpu().numpy(), fs_re.double().cpu().numpy() + 1j * fs_im.double().cpu().numpy()


CASES = [  # (B, T, H, D, N, Q)
    (2, 2048, 16, 64, 64, 64),
    (2, 200, 16, 64, 64, 64),
    (1, 128, 2, 8, 8, 16),
    (2, 333, 4, 40, 16, 32),
    (20, 200, 8, 64, 64, 64),
    (1, 10, 16, 64, 64, 64),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}T{}H{}D{}N{}Q{}".format(*c))
def test_mixer_matches_oracle(case, mimo_path):
    Bn, T, H, D, N, Q = case
    inp = inputs.custom(Bn, T, H, D, N, seed=9000 + T + H)
    W = mixing_matrix(H, 9100 + H)
    y_ref, s_ref = naive_scan_inputs(inp)
    out_ref = head_mix(y_ref, W.astype(np.float64))
    out, s = run_mimo(inp, Q, W, launches=1 if mimo_path == "fused" else 2)
    assert_close(out, s, out_ref, s_ref, "tf32", f"{mimo_path} mixer {case}")


@pytest.mark.parametrize("kernel", [1, 2], ids=["cluster", "tmem"])
def test_identity_mixer_is_the_plain_forward_re_y(lib_option, mimo_path, kernel):
    # the same kernel without the mixer (forced, per-plane tensor maps like the mixer's). The fused
    # epilogue exists on the tensor-memory kernel only: forcing the cluster kernel leaves it there
    on = 2 if mimo_path == "fused" else kernel
    lib_option(ssdc.OPT_FUSED_KERNEL, on)
    lib_option(ssdc.OPT_FUSED_PLANE_MAPS, 0)
    inp = inputs.custom(2, 640, 16, 64, 64, seed=9200)
    t = to_device(inp)
    f = ssdc.Forward(*inp.dims, 64, "tf32")
    y_re, _, fs_re, fs_im = f(*[t[k] for k in ORDER])
    assert ssdc.last_path() == ("fused_cluster" if on == 1 else "fused_tmem")
    lib_option(ssdc.OPT_FUSED_KERNEL, kernel)
    out, s = run_mimo(inp, 64, np.eye(16, dtype=np.float32))
    assert ssdc.last_path() == ("fused_cluster" if on == 1 else "fused_tmem")
    assert np.array_equal(out, y_re.double().cpu().numpy())
    assert np.array_equal(s, fs_re.double().cpu().numpy() + 1j * fs_im.double().cpu().numpy())


def test_mixer_initial_state_and_real_x():
    inp = inputs.custom(2, 300, 8, 64, 64, seed=9300)
    W = mixing_matrix(8, 9301)
    rng = np.random.default_rng(9302)
    Bn, T, H, N, D = inp.dims
    s0 = 8.0 * np.sqrt(0.5) * (rng.standard_normal((Bn, H, N, D)) + 1j * rng.standard_normal((Bn, H, N, D)))
    s0_32 = s0.real.astype(np.float32).astype(np.float64) + 1j * s0.imag.astype(np.float32).astype(np.float64)
    y_ref, s_ref = naive_scan_inputs(inp, s0=s0_32)
    out, s = run_mimo(inp, 64, W, s0=s0)
    assert_close(out, s, head_mix(y_ref, W.astype(np.float64)), s_ref, "tf32", "fused mixer, initial state")
    y_ref, s_ref = naive_scan(inp.x_re, np.zeros_like(inp.x_re), inp.A_re, inp.A_im, inp.B_re, inp.B_im,
                              inp.C_re, inp.C_im, inp.dt)
    out, s = run_mimo(inp, 64, W, real_x=True)
    assert_close(out, s, head_mix(y_ref, W.astype(np.float64)), s_ref, "tf32", "fused mixer, real x")


def test_mixer_rejects_what_it_does_not_take():
    assert ssdc.load().ssd_complex_fwd_mimo_workspace_bytes(ssdc.dims(1, 256, 16, 64, 64, "tf32"), 128) == 0
    assert ssdc.load().ssd_complex_fwd_mimo_workspace_bytes(ssdc.dims(1, 256, 32, 64, 64, "tf32"), 64) == 0
    assert ssdc.load().ssd_complex_fwd_mimo_workspace_bytes(ssdc.dims(1, 256, 16, 64, 64, "fp32"), 64) == 0
    with pytest.raises(ssdc.SSDCError):
        ssdc.MimoForward(1, 256, 16, 64, 64, 128)
