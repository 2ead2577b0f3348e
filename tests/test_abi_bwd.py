"""Host-only checks of the backward entry point (ssd_complex_bwd): workspace
sizes and the rejection of bad arguments before anything reaches a GPU."""
import pytest

from state_space_sequence_complex_gb300 import ssdc


@pytest.fixture(scope="module")
def lib():
    from state_space_sequence_complex_gb300 import build
    build.build()
    return ssdc.load()


# argument order of the fake pointers
IN = ["x_re", "x_im", "A_re", "A_im", "B_re", "B_im", "C_re", "C_im", "dt",
      "s0_re", "s0_im", "dy_re", "dy_im", "dfs_re", "dfs_im"]
OUT = ["dx_re", "dx_im", "dA_re", "dA_im", "dB_re", "dB_im", "dC_re", "dC_im", "ddt",
       "ds0_re", "ds0_im"]
REQUIRED = ["x_re", "A_re", "A_im", "B_re", "B_im", "C_re", "C_im", "dt", "dy_re",
            "dx_re", "dA_re", "dA_im", "dB_re", "dB_im", "dC_re", "dC_im", "ddt"]
PAIRS = [("s0_re", "s0_im"), ("dfs_re", "dfs_im"), ("ds0_re", "ds0_im")]


def sizes(d):
    BTH = d.B * d.T * d.H
    fs = d.B * d.H * d.N * d.D
    return {"x_re": BTH * d.D, "x_im": BTH * d.D, "A_re": d.H, "A_im": d.H,
            "B_re": BTH * d.N, "B_im": BTH * d.N, "C_re": BTH * d.N, "C_im": BTH * d.N,
            "dt": BTH, "s0_re": fs, "s0_im": fs, "dy_re": BTH * d.D, "dy_im": BTH * d.D,
            "dfs_re": fs, "dfs_im": fs, "dx_re": BTH * d.D, "dx_im": BTH * d.D, "dA_re": d.H,
            "dA_im": d.H, "dB_re": BTH * d.N, "dB_im": BTH * d.N, "dC_re": BTH * d.N,
            "dC_im": BTH * d.N, "ddt": BTH, "ds0_re": fs, "ds0_im": fs}


def fake_ptrs(d, base=1 << 32):
    """Distinct, aligned, non-overlapping fake device addresses (never
    dereferenced: each call below stops in its host-side checks, or, with no
    GPU, at the first CUDA call)."""
    out, cur = {}, base
    for k, n in sizes(d).items():
        out[k] = cur
        cur += ((n * 4 + 4095) // 4096) * 4096
    return out, cur


def call(lib, p, d, Q=64, ws=None, ws_bytes=1 << 34):
    cin = lambda a, b: ssdc.ssdc_cin(p[a], p[b])
    cout = lambda a, b: ssdc.ssdc_cout(p[a], p[b])
    return lib.ssd_complex_bwd(cin("x_re", "x_im"), cin("A_re", "A_im"), cin("B_re", "B_im"),
                               cin("C_re", "C_im"), p["dt"], cin("s0_re", "s0_im"),
                               cin("dy_re", "dy_im"), cin("dfs_re", "dfs_im"), d, Q,
                               cout("dx_re", "dx_im"), cout("dA_re", "dA_im"),
                               cout("dB_re", "dB_im"), cout("dC_re", "dC_im"), p["ddt"],
                               cout("ds0_re", "ds0_im"), ws, ws_bytes, None)


PASSED_HOST_CHECKS = (ssdc.SSDC_ERR_CUDA, ssdc.SSDC_ERR_DEVICE)


def no_gpu():
    import torch
    return not torch.cuda.is_available()


def test_workspace_bytes(lib):
    d = ssdc.dims(2, 2048, 16, 64, 64, "fp32")
    chunks = 2 * 16 * 32
    nb = ssdc.ssd_complex_bwd_workspace_bytes(d, 64)
    # chunk states, their gradients, decays, the final state and r_t per token
    assert nb >= 2 * chunks * 2 * 64 * 64 * 4 + chunks * 8 + 2 * 16 * 64 * 64 * 8 + 2 * 2048 * 16 * 8
    # the TF32 backward (Q <= 64) has the same workspace as the exact one
    assert ssdc.ssd_complex_bwd_workspace_bytes(ssdc.dims(2, 2048, 16, 64, 64, "tf32"), 64) == nb
    # at Q = 128 and 256 it works on 64-token chunks: the workspace of Q = 64
    assert ssdc.ssd_complex_bwd_workspace_bytes(ssdc.dims(2, 2048, 16, 64, 64, "tf32"), 128) == nb
    assert ssdc.ssd_complex_bwd_workspace_bytes(ssdc.dims(2, 2048, 16, 64, 64, "tf32"), 256) == nb
    assert ssdc.ssd_complex_bwd_workspace_bytes(ssdc.dims(2, 2048, 16, 64, 64, "fp32"), 128) < nb
    assert ssdc.ssd_complex_bwd_workspace_bytes(ssdc.dims(2, 2048, 16, 64, 64, "tf32"), 48) == 0
    assert ssdc.ssd_complex_bwd_workspace_bytes(ssdc.dims(2, 2048, 16, 12, 64, "tf32"), 64) == 0
    assert ssdc.ssd_complex_bwd_workspace_bytes(ssdc.dims(2, 2048, 16, 64, 64, "tf32_staged"), 64) == 0
    assert ssdc.ssd_complex_bwd_workspace_bytes(ssdc.dims(2, 2048, 16, 64, 64, "fp32"), 48) == 0
    assert ssdc.ssd_complex_bwd_workspace_bytes(ssdc.dims(1, 65, 1, 64, 64, "fp32"), 64) > \
        ssdc.ssd_complex_bwd_workspace_bytes(ssdc.dims(1, 64, 1, 64, 64, "fp32"), 64)


def test_precisions_the_backward_takes(lib):
    """exact fp32 at every size; TF32 at every Q the forward takes (the tensor-core chunk
    gradients, on 64-token chunks above 64); never the staged TF32 precision."""
    d = ssdc.dims(1, 128, 2, 64, 64, "tf32_staged")
    p, end = fake_ptrs(d)
    assert call(lib, p, d, ws=end) == ssdc.SSDC_ERR_UNSUPPORTED
    d = ssdc.dims(1, 128, 2, 64, 64, "tf32")
    p, end = fake_ptrs(d)
    assert call(lib, p, d, Q=48, ws=end) == ssdc.SSDC_ERR_UNSUPPORTED
    for Q in (16, 32, 64, 128, 256):
        assert ssdc.ssd_complex_bwd_workspace_bytes(d, Q) > 0
        if no_gpu():  # passes the host checks (with a GPU it would launch on the fake addresses)
            assert call(lib, p, d, Q=Q, ws=end) in PASSED_HOST_CHECKS


def test_rejects_null_required_pointer(lib):
    d = ssdc.dims(1, 128, 2, 64, 64, "fp32")
    p, end = fake_ptrs(d)
    for k in REQUIRED:
        bad = dict(p, **{k: None})
        assert call(lib, bad, d, ws=end) == ssdc.SSDC_ERR_INVALID, k


def test_rejects_half_pairs_and_equal_planes(lib):
    d = ssdc.dims(1, 128, 2, 64, 64, "fp32")
    p, end = fake_ptrs(d)
    for a, b in PAIRS:
        assert call(lib, dict(p, **{a: None}), d, ws=end) == ssdc.SSDC_ERR_INVALID, a
        assert call(lib, dict(p, **{b: None}), d, ws=end) == ssdc.SSDC_ERR_INVALID, b
        assert call(lib, dict(p, **{b: p[a]}), d, ws=end) == ssdc.SSDC_ERR_INVALID, (a, b)
    assert call(lib, dict(p, x_im=p["x_re"]), d, ws=end) == ssdc.SSDC_ERR_INVALID
    assert call(lib, dict(p, dy_im=p["dy_re"]), d, ws=end) == ssdc.SSDC_ERR_INVALID


def test_rejects_misaligned_pointer(lib):
    d = ssdc.dims(1, 128, 2, 64, 64, "fp32")
    p, end = fake_ptrs(d)
    for k in IN + OUT:
        assert call(lib, dict(p, **{k: p[k] + 4}), d, ws=end) == ssdc.SSDC_ERR_ALIGN, k


def test_rejects_bad_workspace(lib):
    d = ssdc.dims(1, 128, 2, 64, 64, "fp32")
    p, end = fake_ptrs(d)
    need = ssdc.ssd_complex_bwd_workspace_bytes(d, 64)
    assert call(lib, p, d, ws=None) == ssdc.SSDC_ERR_WORKSPACE
    assert call(lib, p, d, ws=end + 16) == ssdc.SSDC_ERR_WORKSPACE
    assert call(lib, p, d, ws=end, ws_bytes=need - 256) == ssdc.SSDC_ERR_WORKSPACE


def test_rejects_overlaps(lib):
    d = ssdc.dims(1, 128, 2, 64, 64, "fp32")
    p, end = fake_ptrs(d)
    for o in OUT:
        for i in IN:
            assert call(lib, dict(p, **{o: p[i]}), d, ws=end) == ssdc.SSDC_ERR_INVALID, (o, i)
        # an output inside the workspace
        assert call(lib, dict(p, **{o: end + 4096}), d, ws=end) == ssdc.SSDC_ERR_INVALID, o
    for a in range(len(OUT)):
        for b in range(a + 1, len(OUT)):
            bad = dict(p, **{OUT[b]: p[OUT[a]]})
            assert call(lib, bad, d, ws=end) == ssdc.SSDC_ERR_INVALID, (OUT[a], OUT[b])


@pytest.mark.skipif("not no_gpu()")
def test_optional_nulls_pass_host_checks(lib):
    """x.im, dy.im, dx.im and the three state pairs may be null: such calls pass
    every host check (without a GPU they then fail at the first CUDA call)."""
    d = ssdc.dims(1, 100, 2, 16, 8, "fp32")
    p, end = fake_ptrs(d)
    opt = dict(p, x_im=None, dy_im=None, dx_im=None, s0_re=None, s0_im=None, dfs_re=None,
               dfs_im=None, ds0_re=None, ds0_im=None)
    assert call(lib, opt, d, Q=32, ws=end) in PASSED_HOST_CHECKS
    assert call(lib, p, d, Q=32, ws=end) in PASSED_HOST_CHECKS


def test_binding_rejects_unsupported_backward_before_allocating(lib):
    """ssdc.Backward raises (no silent fallback) for a precision or size the backward
    does not take, before any device memory is requested."""
    with pytest.raises(ssdc.SSDCError):
        ssdc.Backward(1, 128, 2, 64, 64, 64, precision="tf32_staged", device="cpu")
    with pytest.raises(ssdc.SSDCError):
        ssdc.Backward(1, 128, 2, 64, 64, 48, precision="tf32", device="cpu")
    with pytest.raises(ssdc.SSDCError):
        ssdc.Backward(1, 128, 2, 64, 64, 48, device="cpu")
    with pytest.raises(ssdc.SSDCError):
        ssdc.Backward(1, 128, 2, 72, 64, 64, device="cpu")


def test_header_documents_every_backward_output():
    """Each output of ssd_complex_bwd is described in the header, with its shape."""
    import os
    text = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                             "include", "ssdc.h")).read()
    start = text.index("Backward pass:")
    doc = text[start:text.index("size_t ssd_complex_bwd_workspace_bytes")]
    import re
    for name, shape in (("dx", "(B,T,H,D)"), ("dA", "(H)"), ("dB_t, dC_t", "(B,T,H,N)"),
                        ("ddt", "(B,T,H)"), ("d_initial_state", "(B,H,N,D)")):
        # the argument lines: " *   <name>   output <shape> ..."
        pat = re.compile(r"^\s*\*\s+" + re.escape(name) + r"\s{2,}output")
        line = next(l for l in doc.splitlines() if pat.match(l))
        assert shape in line, (name, line)
