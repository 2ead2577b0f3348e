"""Host-only checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before anything reaches a GPU.

The calls use fake device addresses. A call that passes every host check
would launch kernels on them, so such calls are made only where no GPU is
present (where they then fail at the first CUDA call)."""
import ctypes
import os
import re

import pytest

from state_space_sequence_complex_gb300 import ssdc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssdc.h")


def no_gpu():
    import torch
    return not torch.cuda.is_available()


@pytest.fixture(scope="module")
def lib():
    from state_space_sequence_complex_gb300 import build
    build.build()
    return ssdc.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssd_complex_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 7
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(ssdc.EXPORTS) == names


def test_strerror(lib):
    for code in range(0, -9, -1):
        s = ssdc.strerror(code)
        assert s and s != "unknown status"
    assert ssdc.strerror(-99) == "unknown status"


def test_supported_sets(lib):
    ok = ssdc.ssd_complex_fwd_supported
    assert ok(ssdc.dims(2, 2048, 16, 64, 64, "tf32"), 64) == 0
    assert ok(ssdc.dims(2, 2048, 16, 64, 64, "fp32"), 64) == 0
    assert ok(ssdc.dims(1, 128, 2, 8, 8, "fp32"), 16) == 0
    # TF32: Q = 16 / 32 / 64 / 128 / 256 with N, D multiples of 8 up to 64 (the fused
    # kernels); the staged TF32 path takes N = D = 64 and Q >= 32 only
    assert ok(ssdc.dims(1, 128, 2, 8, 8, "tf32"), 16) == 0
    assert ok(ssdc.dims(1, 128, 2, 8, 24, "tf32"), 32) == 0
    assert ok(ssdc.dims(1, 128, 2, 12, 64, "tf32"), 64) == ssdc.SSDC_ERR_UNSUPPORTED
    assert ok(ssdc.dims(1, 128, 2, 72, 64, "tf32"), 64) == ssdc.SSDC_ERR_UNSUPPORTED
    assert ok(ssdc.dims(1, 128, 2, 32, 64, "tf32"), 128) == 0
    assert ok(ssdc.dims(1, 128, 2, 8, 40, "tf32"), 256) == 0
    assert ok(ssdc.dims(1, 128, 2, 32, 64, "tf32_staged"), 128) == ssdc.SSDC_ERR_UNSUPPORTED
    assert ok(ssdc.dims(1, 128, 2, 64, 64, "tf32"), 512) == ssdc.SSDC_ERR_UNSUPPORTED
    assert ok(ssdc.dims(1, 128, 2, 64, 64, "tf32"), 256) == 0
    assert ok(ssdc.dims(1, 128, 2, 8, 8, "tf32_staged"), 16) == ssdc.SSDC_ERR_UNSUPPORTED
    assert ok(ssdc.dims(1, 128, 2, 64, 64, "fp32"), 48) == ssdc.SSDC_ERR_UNSUPPORTED
    assert ok(ssdc.dims(1, 128, 2, 64, 64, "fp32"), 512) == ssdc.SSDC_ERR_UNSUPPORTED
    assert ok(ssdc.dims(1, 128, 2, 72, 64, "fp32"), 64) == ssdc.SSDC_ERR_UNSUPPORTED
    assert ok(ssdc.dims(1, 128, 2, 12, 64, "fp32"), 64) == ssdc.SSDC_ERR_UNSUPPORTED
    assert ok(ssdc.dims(0, 128, 2, 64, 64, "fp32"), 64) == ssdc.SSDC_ERR_INVALID
    assert ok(ssdc.dims(1, -1, 2, 64, 64, "fp32"), 64) == ssdc.SSDC_ERR_INVALID
    assert ok(ssdc.dims(1, 128, 2, 64, 64, 7), 64) == ssdc.SSDC_ERR_INVALID
    assert ok(ssdc.dims(1, 128, 2, 64, 64, "fp32"), 0) == ssdc.SSDC_ERR_INVALID
    assert ok(ssdc.dims(2, 2048, 16, 64, 64, "tf32_staged"), 64) == 0
    assert ok(ssdc.dims(2, 2048, 16, 64, 64, "tf32_staged"), 32) == 0
    assert ok(ssdc.dims(2, 2048, 16, 64, 64, "tf32"), 32) == 0
    assert ok(ssdc.dims(2, 2048, 16, 64, 64, "tf32_staged"), 16) == ssdc.SSDC_ERR_UNSUPPORTED


def test_workspace_bytes(lib):
    chunks = 2 * 16 * 32
    for prec in ("fp32", "tf32_staged"):
        d = ssdc.dims(2, 2048, 16, 64, 64, prec)
        nb = ssdc.ssd_complex_fwd_workspace_bytes(d, 64)
        assert nb >= chunks * 2 * 64 * 64 * 4 + chunks * 8 + 4
    # the fused tensor-core path keeps the chunk states on chip: status word only
    assert ssdc.ssd_complex_fwd_workspace_bytes(ssdc.dims(2, 2048, 16, 64, 64, "tf32"), 64) == 256
    assert ssdc.ssd_complex_fwd_workspace_bytes(ssdc.dims(1, 128, 2, 8, 8, "tf32"), 16) == 256
    assert ssdc.ssd_complex_fwd_workspace_bytes(ssdc.dims(2, 2048, 16, 64, 64, "tf32"), 32) == 256
    assert ssdc.ssd_complex_fwd_workspace_bytes(ssdc.dims(2, 2048, 16, 64, 64, "tf32"), 128) == 256
    assert ssdc.ssd_complex_fwd_workspace_bytes(ssdc.dims(2, 2048, 16, 64, 64, "tf32"), 256) == 256
    # the staged TF32 path keeps the chunk states in the workspace
    assert ssdc.ssd_complex_fwd_workspace_bytes(ssdc.dims(2, 2048, 16, 64, 64, "tf32_staged"), 128) > 256
    assert ssdc.ssd_complex_fwd_workspace_bytes(ssdc.dims(2, 2048, 16, 64, 64, "tf32"), 48) == 0
    # uneven T rounds the chunk count up
    assert ssdc.ssd_complex_fwd_workspace_bytes(ssdc.dims(1, 65, 1, 64, 64, "fp32"), 64) > \
        ssdc.ssd_complex_fwd_workspace_bytes(ssdc.dims(1, 64, 1, 64, 64, "fp32"), 64)


def _call(lib, ptrs, d, Q=64, ws=None, ws_bytes=1 << 30):
    cin = lambda a, b: ssdc.ssdc_cin(a, b)
    cout = lambda a, b: ssdc.ssdc_cout(a, b)
    p = ptrs
    return lib.ssd_complex_fwd_ws(cin(p[0], p[1]), cin(p[2], p[3]), cin(p[4], p[5]), cin(p[6], p[7]),
                                  p[8], d, Q, cout(p[9], p[10]), cout(p[11], p[12]),
                                  ws, ws_bytes, None)


def fake_ptrs(d, base=1 << 32):
    """Distinct, aligned, non-overlapping fake device addresses (never dereferenced:
    every call below fails its host-side checks before touching the GPU)."""
    BTH = d.B * d.T * d.H
    sizes = [BTH * d.D] * 2 + [d.H] * 2 + [BTH * d.N] * 4 + [BTH] + [BTH * d.D] * 2 + [d.B * d.H * d.N * d.D] * 2
    out, cur = [], base
    for s in sizes:
        out.append(cur)
        cur += ((s * 4 + 4095) // 4096) * 4096
    return out, cur


def test_rejects_null_pointer(lib):
    d = ssdc.dims(1, 128, 2, 64, 64, "fp32")
    ptrs, end = fake_ptrs(d)
    for i in range(13):
        if i == 1:
            continue  # a null x.im means a real x
        bad = list(ptrs)
        bad[i] = None
        assert _call(lib, bad, d, ws=end) == ssdc.SSDC_ERR_INVALID


@pytest.mark.skipif("not no_gpu()")
def test_real_x_passes_argument_checks(lib):
    """x.im = NULL is a real x: it passes the host checks (without a GPU the call then
    fails on the device); x.im equal to x.re is rejected."""
    for prec in ("fp32", "tf32", "tf32_staged"):
        d = ssdc.dims(1, 128, 2, 64, 64, prec)
        ptrs, end = fake_ptrs(d)
        real = list(ptrs)
        real[1] = None
        assert _call(lib, real, d, ws=end) not in (ssdc.SSDC_ERR_INVALID, ssdc.SSDC_ERR_ALIGN,
                                                   ssdc.SSDC_ERR_WORKSPACE, ssdc.SSDC_OK)
        same = list(ptrs)
        same[1] = ptrs[0]
        assert _call(lib, same, d, ws=end) == ssdc.SSDC_ERR_INVALID


def test_rejects_misaligned_pointer(lib):
    d = ssdc.dims(1, 128, 2, 64, 64, "fp32")
    ptrs, end = fake_ptrs(d)
    for i in range(13):
        bad = list(ptrs)
        bad[i] += 4
        assert _call(lib, bad, d, ws=end) == ssdc.SSDC_ERR_ALIGN


def test_rejects_bad_workspace(lib):
    d = ssdc.dims(1, 128, 2, 64, 64, "fp32")
    ptrs, end = fake_ptrs(d)
    need = ssdc.ssd_complex_fwd_workspace_bytes(d, 64)
    assert _call(lib, ptrs, d, ws=None) == ssdc.SSDC_ERR_WORKSPACE
    assert _call(lib, ptrs, d, ws=end + 16) == ssdc.SSDC_ERR_WORKSPACE
    assert _call(lib, ptrs, d, ws=end, ws_bytes=need - 1) == ssdc.SSDC_ERR_WORKSPACE


def test_rejects_overlapping_outputs(lib):
    d = ssdc.dims(1, 128, 2, 64, 64, "fp32")
    ptrs, end = fake_ptrs(d)
    bad = list(ptrs)
    bad[9] = ptrs[0]          # y.re on top of x.re
    assert _call(lib, bad, d, ws=end) == ssdc.SSDC_ERR_INVALID
    bad = list(ptrs)
    bad[12] = ptrs[11]        # final_state planes alias
    assert _call(lib, bad, d, ws=end) == ssdc.SSDC_ERR_INVALID
    bad = list(ptrs)
    bad[9] = end              # y.re inside the workspace
    assert _call(lib, bad, d, ws=end) == ssdc.SSDC_ERR_INVALID


def test_rejects_unsupported_before_launch(lib):
    d = ssdc.dims(1, 128, 2, 64, 64, "tf32_staged")
    ptrs, end = fake_ptrs(d)
    assert _call(lib, ptrs, d, Q=16, ws=end) == ssdc.SSDC_ERR_UNSUPPORTED
    d = ssdc.dims(1, 128, 2, 64, 64, 3)
    assert _call(lib, ptrs, d, ws=end) == ssdc.SSDC_ERR_INVALID


def test_status_null_workspace(lib):
    assert lib.ssd_complex_status(None, None) == ssdc.SSDC_ERR_INVALID


def test_host_scratch_bytes(lib):
    hb = ssdc.ssd_complex_fwd_host_scratch_bytes
    per_token_head = (2 * 64 + 4 * 64 + 1 + 2 * 64) * 4  # x, B, C, dt in; y out
    whole = 2 * 2048 * 16 * per_token_head
    for prec in ("tf32", "fp32"):
        # 134 MB of inputs and outputs, 2 batch rows: 4 segments of 512 tokens of both rows,
        # two on the device at a time (plus, per slot, the final state and, on the fp32
        # path, the staged chunk states)
        nb = hb(ssdc.dims(2, 2048, 16, 64, 64, prec), 64)
        assert 2 * 2 * 512 * 16 * per_token_head <= nb < whole
    # 4.3 GB: 16 groups of 4 batch rows, two on the device at a time
    big = hb(ssdc.dims(64, 2048, 16, 64, 64, "tf32"), 64)
    assert 2 * 4 * 2048 * 16 * per_token_head <= big < 3 * 4 * 2048 * 16 * per_token_head
    assert hb(ssdc.dims(2, 2048, 16, 64, 64, "tf32"), 48) == 0
    assert hb(ssdc.dims(0, 2048, 16, 64, 64, "tf32"), 64) == 0


def _call_host(lib, ptrs, d, Q=64, scratch=None, nbytes=1 << 30):
    cin = lambda a, b: ssdc.ssdc_cin(a, b)
    cout = lambda a, b: ssdc.ssdc_cout(a, b)
    p = ptrs
    return lib.ssd_complex_fwd_host(cin(p[0], p[1]), cin(p[2], p[3]), cin(p[4], p[5]), cin(p[6], p[7]),
                                    p[8], d, Q, cout(p[9], p[10]), cout(p[11], p[12]),
                                    scratch, nbytes, None)


def test_host_entry_rejects_bad_arguments(lib):
    """Host-side checks of the host-buffer entry point: null pointers, overlapping
    outputs, unsupported sizes and a bad scratch buffer, all before any copy."""
    d = ssdc.dims(1, 128, 2, 64, 64, "fp32")
    ptrs, end = fake_ptrs(d)
    scratch = 1 << 44
    for i in range(13):
        if i == 1:
            continue  # a null x.im means a real x
        bad = list(ptrs)
        bad[i] = None
        assert _call_host(lib, bad, d, scratch=scratch) == ssdc.SSDC_ERR_INVALID
    same = list(ptrs)
    same[1] = ptrs[0]
    assert _call_host(lib, same, d, scratch=scratch) == ssdc.SSDC_ERR_INVALID
    for o, i in ((9, 0), (10, 8), (11, 12), (12, 9)):
        bad = list(ptrs)
        bad[o] = ptrs[i]
        assert _call_host(lib, bad, d, scratch=scratch) == ssdc.SSDC_ERR_INVALID
    assert _call_host(lib, ptrs, d, Q=48, scratch=scratch) == ssdc.SSDC_ERR_UNSUPPORTED
    need = ssdc.ssd_complex_fwd_host_scratch_bytes(d, 64)
    assert _call_host(lib, ptrs, d, scratch=None) == ssdc.SSDC_ERR_WORKSPACE
    assert _call_host(lib, ptrs, d, scratch=scratch + 16) == ssdc.SSDC_ERR_WORKSPACE
    assert _call_host(lib, ptrs, d, scratch=scratch, nbytes=need - 1) == ssdc.SSDC_ERR_WORKSPACE


def _call_init(lib, ptrs, s0, d, Q=64, ws=None, ws_bytes=1 << 30):
    cin = lambda a, b: ssdc.ssdc_cin(a, b)
    cout = lambda a, b: ssdc.ssdc_cout(a, b)
    p = ptrs
    return lib.ssd_complex_fwd_init(cin(p[0], p[1]), cin(p[2], p[3]), cin(p[4], p[5]), cin(p[6], p[7]),
                                    p[8], cin(s0[0], s0[1]), d, Q, cout(p[9], p[10]), cout(p[11], p[12]),
                                    ws, ws_bytes, None)


def test_init_entry_rejects_bad_initial_state(lib):
    d = ssdc.dims(1, 128, 2, 64, 64, "fp32")
    ptrs, end = fake_ptrs(d)
    ws = end
    s0 = (end + (4 << 20), end + (8 << 20))  # after the workspace, apart from everything
    need = ssdc.ssd_complex_fwd_workspace_bytes(d, 64)
    call = lambda s: _call_init(lib, ptrs, s, d, ws=ws, ws_bytes=need)
    assert call((s0[0], None)) == ssdc.SSDC_ERR_INVALID          # one plane missing
    assert call((None, s0[1])) == ssdc.SSDC_ERR_INVALID
    assert call((s0[0], s0[0])) == ssdc.SSDC_ERR_INVALID         # one buffer for both planes
    assert call((s0[0] + 4, s0[1])) == ssdc.SSDC_ERR_ALIGN
    assert call((ptrs[9], s0[1])) == ssdc.SSDC_ERR_INVALID       # on top of y.re
    assert call((ws, s0[1])) == ssdc.SSDC_ERR_INVALID            # inside the workspace
    assert call((ptrs[11] + 16, s0[1])) == ssdc.SSDC_ERR_INVALID  # part of the final state
    assert call((ptrs[12], ptrs[11])) == ssdc.SSDC_ERR_INVALID   # the final state's planes swapped
    # the final-state buffer itself (in place) and a separate buffer pass the argument checks;
    # without a GPU the call then fails on the device (with one it would launch)
    if no_gpu():
        for ok in ((ptrs[11], ptrs[12]), s0, (None, None)):
            assert call(ok) not in (ssdc.SSDC_ERR_INVALID, ssdc.SSDC_ERR_ALIGN, ssdc.SSDC_ERR_WORKSPACE)


def test_set_option_rejects_bad_values(lib):
    assert lib.ssd_complex_set_option(ssdc.OPT_FUSED_CLUSTER, 3) == ssdc.SSDC_ERR_INVALID
    assert lib.ssd_complex_set_option(ssdc.OPT_FUSED_PLANE_MAPS, 2) == ssdc.SSDC_ERR_INVALID
    assert lib.ssd_complex_set_option(ssdc.OPT_TEST_DROP_STATE_CHUNK, -2) == ssdc.SSDC_ERR_INVALID
    assert lib.ssd_complex_set_option(ssdc.OPT_MIMO_FUSED, 2) == ssdc.SSDC_ERR_INVALID
    assert lib.ssd_complex_set_option(99, 0) == ssdc.SSDC_ERR_INVALID
    for key, default in ssdc.option.DEFAULTS.items():  # defaults are accepted (and left set)
        assert lib.ssd_complex_set_option(key, default) == ssdc.SSDC_OK


def _call_bf16(lib, ptrs, d, Q=64, ws=None, ws_bytes=1 << 30):
    p = ptrs
    cin = lambda a, b: ssdc.ssdc_cin(a, b)
    cout = lambda a, b: ssdc.ssdc_cout(a, b)
    return lib.ssd_complex_fwd_bf16(cin(p[0], p[1]), cin(p[2], p[3]), cin(p[4], p[5]), cin(p[6], p[7]),
                                    p[8], cin(None, None), d, Q, cout(p[9], p[10]), cout(p[11], p[12]),
                                    ws, ws_bytes, None)


def test_bf16_entry_checks_before_launch(lib):
    """The bfloat16-input entry point takes the TF32 precision and the tensor-memory
    kernel's sizes only; its pointer and overlap checks count 2-byte elements for x, B, C."""
    for prec, N, Q in (("fp32", 64, 64), ("tf32_staged", 64, 64), ("tf32", 12, 64), ("tf32", 64, 48)):
        d = ssdc.dims(1, 128, 2, N, 64, prec)
        ptrs, end = fake_ptrs(d)
        assert _call_bf16(lib, ptrs, d, Q=Q, ws=end) == ssdc.SSDC_ERR_UNSUPPORTED
    d = ssdc.dims(1, 128, 2, 64, 64, "tf32")
    ptrs, end = fake_ptrs(d)
    for i in (0, 2, 4, 8, 9, 12):
        bad = list(ptrs)
        bad[i] = None
        assert _call_bf16(lib, bad, d, ws=end) == ssdc.SSDC_ERR_INVALID
    bad = list(ptrs)
    bad[4] += 8
    assert _call_bf16(lib, bad, d, ws=end) == ssdc.SSDC_ERR_ALIGN
    # y.re starting inside the bfloat16 x.re (its last 16 bytes) is an overlap
    BTH = d.B * d.T * d.H
    inside = list(ptrs)
    inside[9] = ptrs[0] + BTH * d.D * 2 - 16
    assert _call_bf16(lib, inside, d, ws=end) == ssdc.SSDC_ERR_INVALID


def _call_mimo(lib, ptrs, mix, d, Q=64, ws=None, ws_bytes=1 << 30):
    p = ptrs
    cin = lambda a, b: ssdc.ssdc_cin(a, b)
    cout = lambda a, b: ssdc.ssdc_cout(a, b)
    return lib.ssd_complex_fwd_mimo(cin(p[0], p[1]), cin(p[2], p[3]), cin(p[4], p[5]), cin(p[6], p[7]),
                                    p[8], mix, cin(None, None), d, Q, p[9], cout(p[11], p[12]),
                                    ws, ws_bytes, None)


def test_mimo_entry_checks_before_launch(lib):
    """The fused head mixer takes the TF32 precision, Q <= 64 and H <= 16; the matrix is required,
    must be aligned and must not overlap an output; its workspace holds the tile counters."""
    d = ssdc.dims(2, 128, 16, 64, 64, "tf32")
    ptrs, end = fake_ptrs(d)
    mix = end + (1 << 20)
    need = lib.ssd_complex_fwd_mimo_workspace_bytes(d, 64)
    assert need >= 256 + 4 * 2 * 2
    assert _call_mimo(lib, ptrs, None, d, ws=end) == ssdc.SSDC_ERR_INVALID
    assert _call_mimo(lib, ptrs, mix + 4, d, ws=end) == ssdc.SSDC_ERR_ALIGN
    assert _call_mimo(lib, ptrs, ptrs[9], d, ws=end) == ssdc.SSDC_ERR_INVALID       # on top of out
    assert _call_mimo(lib, ptrs, mix, d, ws=end, ws_bytes=need - 1) == ssdc.SSDC_ERR_WORKSPACE
    for prec, H, Q in (("fp32", 16, 64), ("tf32", 16, 128), ("tf32", 32, 64)):
        dd = ssdc.dims(2, 128, H, 64, 64, prec)
        p2, e2 = fake_ptrs(dd)
        assert _call_mimo(lib, p2, e2 + (1 << 20), dd, Q=Q, ws=e2) == ssdc.SSDC_ERR_UNSUPPORTED
    if no_gpu():  # passes the host checks (with a GPU it would launch)
        assert _call_mimo(lib, ptrs, mix, d, ws=end, ws_bytes=need) not in (
            ssdc.SSDC_ERR_INVALID, ssdc.SSDC_ERR_ALIGN, ssdc.SSDC_ERR_WORKSPACE, ssdc.SSDC_OK)


def _call_state(lib, ptrs, d, s0=(None, None), Q=64, ws=None, ws_bytes=1 << 30):
    # ptrs in fake_ptrs order: x (0, 1), A (2, 3), B (4, 5), C (6, 7), dt (8), y (9, 10), final state (11, 12)
    p = ptrs
    cin = lambda a, b: ssdc.ssdc_cin(a, b)
    return lib.ssd_complex_final_state(cin(p[0], p[1]), cin(p[2], p[3]), cin(p[4], p[5]), p[8], cin(*s0), d, Q,
                                       ssdc.ssdc_cout(p[11], p[12]), ws, ws_bytes, None)


def test_final_state_entry_checks_before_launch(lib):
    """ssd_complex_final_state: the forward's size sets, its workspace (the status word on the
    TF32 path, the chunk states on the staged ones), every required pointer, 16-byte alignment,
    no output overlapping an input or the workspace, and an initial state that is either apart
    from the final state or the final state itself."""
    d = ssdc.dims(2, 128, 4, 64, 64, "tf32")
    ptrs, end = fake_ptrs(d)
    need = lib.ssd_complex_final_state_workspace_bytes(d, 64)
    assert need == 256
    assert lib.ssd_complex_final_state_workspace_bytes(ssdc.dims(2, 128, 4, 64, 64, "fp32"), 64) == \
        lib.ssd_complex_fwd_workspace_bytes(ssdc.dims(2, 128, 4, 64, 64, "fp32"), 64)
    assert lib.ssd_complex_final_state_workspace_bytes(ssdc.dims(2, 128, 4, 64, 64, "tf32"), 48) == 0
    call = lambda p=ptrs, **kw: _call_state(lib, p, d, ws=kw.pop("ws", end), **kw)
    for i in (0, 2, 3, 4, 5, 8, 11, 12):  # x.re, A, B, dt, the final state
        bad = list(ptrs)
        bad[i] = None
        assert call(bad) == ssdc.SSDC_ERR_INVALID, i
    bad = list(ptrs)
    bad[4] += 4
    assert call(bad) == ssdc.SSDC_ERR_ALIGN
    assert call(ws=None) == ssdc.SSDC_ERR_WORKSPACE
    assert call(ws_bytes=need - 1) == ssdc.SSDC_ERR_WORKSPACE
    bad = list(ptrs)
    bad[11] = ptrs[4]  # the final state on top of B
    assert call(bad) == ssdc.SSDC_ERR_INVALID
    bad = list(ptrs)
    bad[12] = ptrs[11] + 16  # its planes overlapping
    assert call(bad) == ssdc.SSDC_ERR_INVALID
    s0 = (end + (4 << 20), end + (8 << 20))
    assert call(s0=(s0[0], None)) == ssdc.SSDC_ERR_INVALID
    assert call(s0=(ptrs[11] + 16, s0[1])) == ssdc.SSDC_ERR_INVALID  # part of the final state
    assert call(s0=(end, s0[1])) == ssdc.SSDC_ERR_INVALID            # inside the workspace
    assert _call_state(lib, ptrs, d, Q=48, ws=end) == ssdc.SSDC_ERR_UNSUPPORTED
    # C and y are not arguments: their fake addresses may hold anything; a real x, the final
    # state as its own initial state and a separate one pass the argument checks (without a GPU
    # the call then fails on the device; with one it would launch)
    real = list(ptrs)
    real[1] = None
    for p, s in ((real, (None, None)), (ptrs, (ptrs[11], ptrs[12])), (ptrs, s0)):
        if no_gpu():
            assert _call_state(lib, p, d, s0=s, ws=end, ws_bytes=need) not in (
                ssdc.SSDC_ERR_INVALID, ssdc.SSDC_ERR_ALIGN, ssdc.SSDC_ERR_WORKSPACE, ssdc.SSDC_OK)
