"""Thin ctypes binding of libssdc.so (include/ssdc.h): argument marshalling only.

Every step of the scan runs in the library's CUDA kernels. PyTorch supplies
device memory and the current stream. There is no fallback: if the library is
missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libssdc.so")

SSDC_OK = 0
SSDC_ERR_INVALID = -1
SSDC_ERR_UNSUPPORTED = -2
SSDC_ERR_ALIGN = -3
SSDC_ERR_WORKSPACE = -4
SSDC_ERR_CUDA = -5
SSDC_ERR_TIMEOUT = -6
SSDC_ERR_DEVICE = -7
SSDC_ERR_TOO_LARGE = -8
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024 + 64 * 1024

PREC = {"tf32": 0, "fp32": 1, "tf32_staged": 2}

# Every symbol include/ssdc.h declares.
EXPORTS = ("ssd_complex_fwd_supported", "ssd_complex_fwd_workspace_bytes", "ssd_complex_fwd_ws",
           "ssd_complex_fwd", "ssd_complex_status", "ssd_complex_strerror",
           "ssd_complex_last_launch_count", "ssd_complex_timing_enable", "ssd_complex_timing_read",
           "ssd_complex_fwd_noalloc", "ssd_complex_fwd_host_scratch_bytes", "ssd_complex_fwd_host",
           "ssd_complex_fwd_init", "ssd_complex_bwd_workspace_bytes", "ssd_complex_bwd",
           "ssd_complex_set_option", "ssd_complex_noalloc_status", "ssd_complex_last_path",
           "ssd_complex_segment_decay", "ssd_complex_state_combine", "ssd_complex_fwd_bf16",
           "ssd_complex_fwd_mimo", "ssd_complex_fwd_mimo_workspace_bytes", "ssd_complex_final_state",
           "ssd_complex_final_state_workspace_bytes")

PATHS = {0: "staged_fp32", 1: "staged_tf32", 2: "fused_cluster", 3: "fused_tmem", 4: "state_tmem"}

# ssd_complex_set_option keys
OPT_FUSED_CLUSTER = 1
OPT_FUSED_PLANE_MAPS = 2
OPT_TEST_DROP_STATE_CHUNK = 3
OPT_FUSED_KERNEL = 4
OPT_MIMO_FUSED = 5


class ssdc_dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("T", ctypes.c_int64), ("H", ctypes.c_int64),
                ("N", ctypes.c_int64), ("D", ctypes.c_int64), ("precision", ctypes.c_int32)]


class ssdc_cin(ctypes.Structure):
    _fields_ = [("re", ctypes.c_void_p), ("im", ctypes.c_void_p)]


class ssdc_cout(ctypes.Structure):
    _fields_ = [("re", ctypes.c_void_p), ("im", ctypes.c_void_p)]


class SSDCError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {strerror(status)} (status {status})")
        self.status = status


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Open libssdc.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise FileNotFoundError(f"{path} is missing: build it with __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    lib.ssd_complex_fwd_supported.argtypes = [ssdc_dims, ctypes.c_int]
    lib.ssd_complex_fwd_supported.restype = ctypes.c_int
    lib.ssd_complex_fwd_workspace_bytes.argtypes = [ssdc_dims, ctypes.c_int]
    lib.ssd_complex_fwd_workspace_bytes.restype = sz
    common = [ssdc_cin, ssdc_cin, ssdc_cin, ssdc_cin, vp, ssdc_dims, ctypes.c_int, ssdc_cout, ssdc_cout]
    lib.ssd_complex_fwd_ws.argtypes = common + [vp, sz, vp]
    lib.ssd_complex_fwd_ws.restype = ctypes.c_int
    lib.ssd_complex_fwd_init.argtypes = common[:5] + [ssdc_cin] + common[5:] + [vp, sz, vp]
    lib.ssd_complex_fwd_init.restype = ctypes.c_int
    lib.ssd_complex_fwd_bf16.argtypes = common[:5] + [ssdc_cin] + common[5:] + [vp, sz, vp]
    lib.ssd_complex_fwd_bf16.restype = ctypes.c_int
    lib.ssd_complex_fwd_mimo.argtypes = common[:5] + [vp, ssdc_cin, ssdc_dims, ctypes.c_int, vp, ssdc_cout,
                                                      vp, sz, vp]
    lib.ssd_complex_fwd_mimo.restype = ctypes.c_int
    lib.ssd_complex_fwd_mimo_workspace_bytes.argtypes = [ssdc_dims, ctypes.c_int]
    lib.ssd_complex_fwd_mimo_workspace_bytes.restype = sz
    lib.ssd_complex_fwd.argtypes = common + [vp]
    lib.ssd_complex_fwd.restype = ctypes.c_int
    lib.ssd_complex_status.argtypes = [vp, vp]
    lib.ssd_complex_status.restype = ctypes.c_int
    lib.ssd_complex_strerror.argtypes = [ctypes.c_int]
    lib.ssd_complex_strerror.restype = ctypes.c_char_p
    lib.ssd_complex_last_launch_count.argtypes = []
    lib.ssd_complex_last_launch_count.restype = ctypes.c_int
    lib.ssd_complex_fwd_noalloc.argtypes = common + [vp]
    lib.ssd_complex_fwd_noalloc.restype = ctypes.c_int
    lib.ssd_complex_fwd_host_scratch_bytes.argtypes = [ssdc_dims, ctypes.c_int]
    lib.ssd_complex_fwd_host_scratch_bytes.restype = sz
    lib.ssd_complex_fwd_host.argtypes = common + [vp, sz, vp]
    lib.ssd_complex_fwd_host.restype = ctypes.c_int
    lib.ssd_complex_bwd_workspace_bytes.argtypes = [ssdc_dims, ctypes.c_int]
    lib.ssd_complex_bwd_workspace_bytes.restype = sz
    lib.ssd_complex_bwd.argtypes = ([ssdc_cin] * 4 + [vp] + [ssdc_cin] * 3 + [ssdc_dims, ctypes.c_int]
                                    + [ssdc_cout] * 4 + [vp, ssdc_cout, vp, sz, vp])
    lib.ssd_complex_bwd.restype = ctypes.c_int
    lib.ssd_complex_timing_enable.argtypes = [ctypes.c_int]
    lib.ssd_complex_timing_enable.restype = ctypes.c_int
    lib.ssd_complex_timing_read.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_int]
    lib.ssd_complex_timing_read.restype = ctypes.c_int
    lib.ssd_complex_set_option.argtypes = [ctypes.c_int, ctypes.c_int64]
    lib.ssd_complex_set_option.restype = ctypes.c_int
    lib.ssd_complex_segment_decay.argtypes = [ssdc_cin, vp, ssdc_dims, ssdc_cout, vp]
    lib.ssd_complex_final_state.argtypes = [ssdc_cin, ssdc_cin, ssdc_cin, vp, ssdc_cin, ssdc_dims, ctypes.c_int,
                                            ssdc_cout, vp, sz, vp]
    lib.ssd_complex_final_state.restype = ctypes.c_int
    lib.ssd_complex_final_state_workspace_bytes.argtypes = [ssdc_dims, ctypes.c_int]
    lib.ssd_complex_final_state_workspace_bytes.restype = sz
    lib.ssd_complex_segment_decay.restype = ctypes.c_int
    lib.ssd_complex_state_combine.argtypes = [ssdc_cin, ssdc_cin, ssdc_cin, ssdc_dims, ssdc_cout, vp]
    lib.ssd_complex_state_combine.restype = ctypes.c_int
    lib.ssd_complex_last_path.argtypes = []
    lib.ssd_complex_last_path.restype = ctypes.c_int
    lib.ssd_complex_noalloc_status.argtypes = [vp]
    lib.ssd_complex_noalloc_status.restype = ctypes.c_int
    _lib = lib
    return lib


def strerror(status: int) -> str:
    return load().ssd_complex_strerror(int(status)).decode()


def dims(Bn, T, H, N, D, precision="tf32") -> ssdc_dims:
    return ssdc_dims(int(Bn), int(T), int(H), int(N), int(D), PREC[precision] if isinstance(precision, str) else int(precision))


def ssd_complex_fwd_supported(d: ssdc_dims, chunk_size: int) -> int:
    return load().ssd_complex_fwd_supported(d, int(chunk_size))


def ssd_complex_fwd_workspace_bytes(d: ssdc_dims, chunk_size: int) -> int:
    return int(load().ssd_complex_fwd_workspace_bytes(d, int(chunk_size)))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _cin(re, im):
    """Planar input; ``im`` may be None for a real x."""
    return ssdc_cin(re.data_ptr(), None if im is None else im.data_ptr())


def _cout(re, im):
    return ssdc_cout(re.data_ptr(), im.data_ptr())


def _opt_in(re, im):
    """Planar input where either plane may be None (a null pointer)."""
    return ssdc_cin(None if re is None else re.data_ptr(), None if im is None else im.data_ptr())


def _opt_out(re, im):
    return ssdc_cout(None if re is None else re.data_ptr(), None if im is None else im.data_ptr())


def ssd_complex_fwd_ws(x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt, chunk_size, *,
                       precision="tf32", y_re, y_im, fs_re, fs_im, workspace, stream=None,
                       check=True) -> int:
    """Call ``ssd_complex_fwd_ws`` on torch CUDA tensors (planar float32).

    ``workspace`` is a uint8 CUDA tensor of at least the queried size;
    ``stream`` a ``torch.cuda.Stream`` (default: the current stream).
    Returns the status (raises on a non-zero one unless ``check`` is False).
    """
    import torch

    Bn, T, H, D = x_re.shape
    N = B_re.shape[-1]
    d = dims(Bn, T, H, N, D, precision)
    s = torch.cuda.current_stream() if stream is None else stream
    rc = load().ssd_complex_fwd_ws(
        _cin(x_re, x_im), _cin(A_re, A_im), _cin(B_re, B_im), _cin(C_re, C_im), _ptr(dt), d,
        int(chunk_size), _cout(y_re, y_im), _cout(fs_re, fs_im), _ptr(workspace),
        int(workspace.numel()), ctypes.c_void_p(s.cuda_stream))
    if check and rc != SSDC_OK:
        raise SSDCError(rc, "ssd_complex_fwd_ws")
    return rc


def ssd_complex_fwd_init(x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt, s0_re, s0_im, chunk_size, *,
                         precision="tf32", y_re, y_im, fs_re, fs_im, workspace, stream=None,
                         check=True) -> int:
    """Call ``ssd_complex_fwd_init`` on torch CUDA tensors: the forward pass from
    the initial state (s0_re, s0_im) of shape (B,H,N,D) (None, None: zero). The
    initial state may be the (fs_re, fs_im) tensors themselves. Returns the status."""
    import torch

    Bn, T, H, D = x_re.shape
    N = B_re.shape[-1]
    d = dims(Bn, T, H, N, D, precision)
    s = torch.cuda.current_stream() if stream is None else stream
    s0 = ssdc_cin(None if s0_re is None else s0_re.data_ptr(), None if s0_im is None else s0_im.data_ptr())
    rc = load().ssd_complex_fwd_init(
        _cin(x_re, x_im), _cin(A_re, A_im), _cin(B_re, B_im), _cin(C_re, C_im), _ptr(dt), s0, d,
        int(chunk_size), _cout(y_re, y_im), _cout(fs_re, fs_im), _ptr(workspace),
        int(workspace.numel()), ctypes.c_void_p(s.cuda_stream))
    if check and rc != SSDC_OK:
        raise SSDCError(rc, "ssd_complex_fwd_init")
    return rc


def ssd_complex_fwd_bf16(x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt, chunk_size, *, s0_re=None,
                         s0_im=None, y_re, y_im, fs_re, fs_im, workspace, stream=None, check=True) -> int:
    """Call ``ssd_complex_fwd_bf16`` on torch CUDA tensors: x, B, C planar
    ``torch.bfloat16`` (``x_im`` may be None for a real x); A, dt, the optional
    initial state (s0_re, s0_im) and the outputs float32. Returns the status."""
    import torch

    for t in (x_re, x_im, B_re, B_im, C_re, C_im):
        if t is not None and t.dtype != torch.bfloat16:
            raise TypeError("x, B and C must be torch.bfloat16")
    Bn, T, H, D = x_re.shape
    N = B_re.shape[-1]
    d = dims(Bn, T, H, N, D, "tf32")
    s = torch.cuda.current_stream() if stream is None else stream
    rc = load().ssd_complex_fwd_bf16(
        _cin(x_re, x_im), _cin(A_re, A_im), _cin(B_re, B_im), _cin(C_re, C_im), _ptr(dt), _opt_in(s0_re, s0_im),
        d, int(chunk_size), _cout(y_re, y_im), _cout(fs_re, fs_im), _ptr(workspace), int(workspace.numel()),
        ctypes.c_void_p(s.cuda_stream))
    if check and rc != SSDC_OK:
        raise SSDCError(rc, "ssd_complex_fwd_bf16")
    return rc


class MimoForward:
    """The forward pass followed by the MIMO head mixer (``ssd_complex_fwd_mimo``:
    the scan writes Re(y) into the output and a second kernel mixes it in place,
    or with ``OPT_MIMO_FUSED`` = 1 the mixer runs in the scan's epilogue): holds the output (the mixed Re(y), (B,T,H,D)), the final state and the
    workspace of one problem size. ``__call__`` takes the planar inputs and the
    (H,H) mixing matrix as CUDA tensors and returns ``(out, fs_re, fs_im)``."""

    def __init__(self, Bn, T, H, N, D, chunk_size, device="cuda"):
        import torch

        self.shape = (Bn, T, H, N, D)
        self.chunk_size = int(chunk_size)
        d = dims(Bn, T, H, N, D, "tf32")
        nbytes = load().ssd_complex_fwd_mimo_workspace_bytes(d, int(chunk_size))
        if nbytes == 0:
            raise SSDCError(SSDC_ERR_UNSUPPORTED, "ssd_complex_fwd_mimo_workspace_bytes")
        f32 = dict(dtype=torch.float32, device=device)
        self.out = torch.empty((Bn, T, H, D), **f32)
        self.fs_re = torch.empty((Bn, H, N, D), **f32)
        self.fs_im = torch.empty((Bn, H, N, D), **f32)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)

    def __call__(self, x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt, mix, stream=None, s0_re=None,
                 s0_im=None):
        import torch

        Bn, T, H, N, D = self.shape
        s = torch.cuda.current_stream() if stream is None else stream
        rc = load().ssd_complex_fwd_mimo(
            _cin(x_re, x_im), _cin(A_re, A_im), _cin(B_re, B_im), _cin(C_re, C_im), _ptr(dt), _ptr(mix),
            _opt_in(s0_re, s0_im), dims(Bn, T, H, N, D, "tf32"), self.chunk_size, _ptr(self.out),
            _cout(self.fs_re, self.fs_im), _ptr(self.workspace), int(self.workspace.numel()),
            ctypes.c_void_p(s.cuda_stream))
        if rc != SSDC_OK:
            raise SSDCError(rc, "ssd_complex_fwd_mimo")
        return self.out, self.fs_re, self.fs_im

    def status(self, stream=None) -> int:
        return ssd_complex_status(self.workspace, stream)


def ssd_complex_fwd_noalloc(x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt, chunk_size, *,
                            precision="fp32", y_re, y_im, fs_re, fs_im, stream=None, check=True) -> int:
    """Call ``ssd_complex_fwd_noalloc`` on torch CUDA tensors: the staged path
    with the library's static scratch workspace, for callers that cannot
    allocate device memory while they run the scan. Returns the status."""
    import torch

    Bn, T, H, D = x_re.shape
    N = B_re.shape[-1]
    d = dims(Bn, T, H, N, D, precision)
    s = torch.cuda.current_stream() if stream is None else stream
    rc = load().ssd_complex_fwd_noalloc(
        _cin(x_re, x_im), _cin(A_re, A_im), _cin(B_re, B_im), _cin(C_re, C_im), _ptr(dt), d,
        int(chunk_size), _cout(y_re, y_im), _cout(fs_re, fs_im), ctypes.c_void_p(s.cuda_stream))
    if check and rc != SSDC_OK:
        raise SSDCError(rc, "ssd_complex_fwd_noalloc")
    return rc


def ssd_complex_fwd_host_scratch_bytes(d: ssdc_dims, chunk_size: int) -> int:
    return int(load().ssd_complex_fwd_host_scratch_bytes(d, int(chunk_size)))


def ssd_complex_fwd_host(x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt, chunk_size, *,
                         precision="tf32", y_re, y_im, fs_re, fs_im, scratch, stream=None,
                         check=True) -> int:
    """Call ``ssd_complex_fwd_host``: inputs and outputs are contiguous float32
    CPU tensors (pinned for overlapped copies), ``scratch`` a uint8 CUDA tensor
    of at least ``ssd_complex_fwd_host_scratch_bytes`` bytes. Returns when the
    outputs are in the host tensors, with the status."""
    import torch

    Bn, T, H, D = x_re.shape
    N = B_re.shape[-1]
    d = dims(Bn, T, H, N, D, precision)
    s = torch.cuda.current_stream() if stream is None else stream
    rc = load().ssd_complex_fwd_host(
        _cin(x_re, x_im), _cin(A_re, A_im), _cin(B_re, B_im), _cin(C_re, C_im), _ptr(dt), d,
        int(chunk_size), _cout(y_re, y_im), _cout(fs_re, fs_im), _ptr(scratch),
        int(scratch.numel()), ctypes.c_void_p(s.cuda_stream))
    if check and rc != SSDC_OK:
        raise SSDCError(rc, "ssd_complex_fwd_host")
    return rc


def ssd_complex_bwd_workspace_bytes(d: ssdc_dims, chunk_size: int) -> int:
    return int(load().ssd_complex_bwd_workspace_bytes(d, int(chunk_size)))


def ssd_complex_bwd(x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt, chunk_size, *,
                    dy_re, dy_im=None, dfs_re=None, dfs_im=None, s0_re=None, s0_im=None,
                    dx_re, dx_im=None, dA_re, dA_im, dB_re, dB_im, dC_re, dC_im, ddt,
                    ds0_re=None, ds0_im=None, workspace, precision="fp32", stream=None,
                    check=True) -> int:
    """Call ``ssd_complex_bwd`` on torch CUDA tensors (planar float32): the
    gradients of every input given ``dy`` (and ``dfs``, the gradient of the
    final state; None: zero). ``x_im``, ``dy_im`` and ``dx_im`` may be None;
    ``s0``, ``dfs`` and ``ds0`` are pairs given together or not at all.
    Returns the status (raises on a non-zero one unless ``check`` is False)."""
    import torch

    Bn, T, H, D = x_re.shape
    N = B_re.shape[-1]
    d = dims(Bn, T, H, N, D, precision)
    s = torch.cuda.current_stream() if stream is None else stream
    rc = load().ssd_complex_bwd(
        _cin(x_re, x_im), _cin(A_re, A_im), _cin(B_re, B_im), _cin(C_re, C_im), _ptr(dt),
        _opt_in(s0_re, s0_im), _opt_in(dy_re, dy_im), _opt_in(dfs_re, dfs_im), d, int(chunk_size),
        _opt_out(dx_re, dx_im), _cout(dA_re, dA_im), _cout(dB_re, dB_im), _cout(dC_re, dC_im),
        _ptr(ddt), _opt_out(ds0_re, ds0_im), _ptr(workspace), int(workspace.numel()),
        ctypes.c_void_p(s.cuda_stream))
    if check and rc != SSDC_OK:
        raise SSDCError(rc, "ssd_complex_bwd")
    return rc


class Backward:
    """Holds the input gradients and the workspace of one problem size, so
    repeated backward calls allocate nothing. ``__call__`` takes the forward
    inputs and the output gradients as CUDA tensors and returns a dict of
    gradients: ``dx_re``, ``dx_im``, ``dA_re``, ``dA_im``, ``dB_re``, ``dB_im``,
    ``dC_re``, ``dC_im``, ``ddt`` and, with an initial state, ``ds0_re`` and
    ``ds0_im``."""

    def __init__(self, Bn, T, H, N, D, chunk_size, precision="fp32", device="cuda"):
        import torch

        self.shape = (Bn, T, H, N, D)
        self.chunk_size = int(chunk_size)
        self.precision = precision
        d = dims(Bn, T, H, N, D, precision)
        nbytes = ssd_complex_bwd_workspace_bytes(d, chunk_size)
        if nbytes == 0:
            raise SSDCError(SSDC_ERR_UNSUPPORTED, "ssd_complex_bwd_workspace_bytes")
        f32 = dict(dtype=torch.float32, device=device)
        self.grads = {
            "dx_re": torch.empty((Bn, T, H, D), **f32), "dx_im": torch.empty((Bn, T, H, D), **f32),
            "dA_re": torch.empty((H,), **f32), "dA_im": torch.empty((H,), **f32),
            "dB_re": torch.empty((Bn, T, H, N), **f32), "dB_im": torch.empty((Bn, T, H, N), **f32),
            "dC_re": torch.empty((Bn, T, H, N), **f32), "dC_im": torch.empty((Bn, T, H, N), **f32),
            "ddt": torch.empty((Bn, T, H), **f32),
            "ds0_re": torch.empty((Bn, H, N, D), **f32), "ds0_im": torch.empty((Bn, H, N, D), **f32)}
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)

    def __call__(self, x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt, dy_re, dy_im=None,
                 dfs_re=None, dfs_im=None, s0_re=None, s0_im=None, stream=None):
        g = self.grads
        with_s0 = s0_re is not None
        ssd_complex_bwd(x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt, self.chunk_size,
                        dy_re=dy_re, dy_im=dy_im, dfs_re=dfs_re, dfs_im=dfs_im, s0_re=s0_re,
                        s0_im=s0_im, dx_re=g["dx_re"], dx_im=None if x_im is None else g["dx_im"],
                        dA_re=g["dA_re"], dA_im=g["dA_im"], dB_re=g["dB_re"], dB_im=g["dB_im"],
                        dC_re=g["dC_re"], dC_im=g["dC_im"], ddt=g["ddt"],
                        ds0_re=g["ds0_re"] if with_s0 else None,
                        ds0_im=g["ds0_im"] if with_s0 else None,
                        workspace=self.workspace, precision=self.precision, stream=stream)
        out = {k: v for k, v in g.items() if not k.startswith("ds0") or with_s0}
        if x_im is None:
            out.pop("dx_im")
        return out


def _scan_function():
    """The torch.autograd.Function over the library's forward and backward
    passes (built on first use so that importing this module needs no torch)."""
    import torch

    class SSDComplexScan(torch.autograd.Function):
        """Forward: ``ssd_complex_fwd_ws`` / ``_init``. Backward: ``ssd_complex_bwd``,
        seeded with the true gradients of all four outputs (zeros where autograd
        passes None), returning a gradient for every tensor input."""

        @staticmethod
        def forward(ctx, chunk_size, precision, bwd_precision, x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im,
                    dt, s0_re, s0_im):
            Bn, T, H, D = x_re.shape
            N = B_re.shape[-1]
            f = Forward(Bn, T, H, N, D, chunk_size, precision, device=x_re.device)
            y_re, y_im, fs_re, fs_im = f(x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt,
                                         s0_re=s0_re, s0_im=s0_im)
            ctx.chunk_size = chunk_size
            ctx.bwd_precision = bwd_precision
            ctx.real_x = x_im is None
            ctx.with_s0 = s0_re is not None
            ctx.save_for_backward(x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt, s0_re, s0_im)
            return y_re, y_im, fs_re, fs_im

        @staticmethod
        def backward(ctx, gy_re, gy_im, gfs_re, gfs_im):
            x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt, s0_re, s0_im = ctx.saved_tensors
            Bn, T, H, D = x_re.shape
            N = B_re.shape[-1]
            z = lambda shape: torch.zeros(shape, dtype=torch.float32, device=x_re.device)
            gy_re = z((Bn, T, H, D)) if gy_re is None else gy_re.contiguous()
            gy_im = None if gy_im is None else gy_im.contiguous()
            if gfs_re is None and gfs_im is None:
                gfs = (None, None)
            else:
                gfs = (z((Bn, H, N, D)) if gfs_re is None else gfs_re.contiguous(),
                       z((Bn, H, N, D)) if gfs_im is None else gfs_im.contiguous())
            b = Backward(Bn, T, H, N, D, ctx.chunk_size, ctx.bwd_precision, device=x_re.device)
            g = b(x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt, gy_re, gy_im, *gfs,
                  s0_re=s0_re if ctx.with_s0 else None, s0_im=s0_im if ctx.with_s0 else None)
            return (None, None, None, g["dx_re"], None if ctx.real_x else g["dx_im"], g["dA_re"],
                    g["dA_im"], g["dB_re"], g["dB_im"], g["dC_re"], g["dC_im"], g["ddt"],
                    g["ds0_re"] if ctx.with_s0 else None, g["ds0_im"] if ctx.with_s0 else None)

    return SSDComplexScan


_SCAN_FN = None


def ssd_complex_scan(x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt, chunk_size, *,
                     s0_re=None, s0_im=None, precision="tf32", bwd_precision="fp32"):
    """Differentiable complex SSD scan on planar float32 CUDA tensors: returns
    ``(y_re, y_im, final_state_re, final_state_im)``; ``y_re`` is Re(y). The
    forward runs at ``precision``; the backward is the library's backward pass
    at ``bwd_precision`` ("fp32": exact; "tf32": the chunk gradients on the
    tensor cores, chunk sizes up to 64). ``x_im`` may be None (a real x); the
    initial state ``(s0_re, s0_im)`` is optional."""
    global _SCAN_FN
    if _SCAN_FN is None:
        _SCAN_FN = _scan_function()
    return _SCAN_FN.apply(int(chunk_size), precision, bwd_precision, x_re, x_im, A_re, A_im, B_re, B_im,
                          C_re, C_im, dt, s0_re, s0_im)


def ssd_complex_status(workspace, stream=None) -> int:
    import torch

    s = torch.cuda.current_stream() if stream is None else stream
    return load().ssd_complex_status(_ptr(workspace), ctypes.c_void_p(s.cuda_stream))


def ssd_complex_segment_decay(A_re, A_im, dt, *, a_re, a_im, stream=None) -> None:
    """a_seg[b,h] = exp(sum_t softplus(dt[b,t,h]) A[h]) into (a_re, a_im) (B,H)."""
    import torch
    Bn, T, H = dt.shape
    s = torch.cuda.current_stream() if stream is None else stream
    rc = load().ssd_complex_segment_decay(_cin(A_re, A_im), _ptr(dt), dims(Bn, T, H, 1, 1, "fp32"),
                                          _cout(a_re, a_im), ctypes.c_void_p(s.cuda_stream))
    if rc != SSDC_OK:
        raise SSDCError(rc, "ssd_complex_segment_decay")


def ssd_complex_final_state(x_re, x_im, A_re, A_im, B_re, B_im, dt, chunk_size, *, precision="tf32",
                            s0_re=None, s0_im=None, fs_re, fs_im, workspace, stream=None, check=True) -> int:
    """Call ``ssd_complex_final_state`` on torch CUDA tensors: the state the scan of
    (x, A, B_t, dt) leaves, from the initial state (s0_re, s0_im) (None, None: zero),
    into (fs_re, fs_im) (B,H,N,D), without y. ``workspace``: a uint8 CUDA tensor of
    ``ssd_complex_final_state_workspace_bytes`` bytes. Returns the status."""
    import torch
    Bn, T, H, D = x_re.shape
    N = B_re.shape[-1]
    s = torch.cuda.current_stream() if stream is None else stream
    rc = load().ssd_complex_final_state(
        _cin(x_re, x_im), _cin(A_re, A_im), _cin(B_re, B_im), _ptr(dt), _opt_in(s0_re, s0_im),
        dims(Bn, T, H, N, D, precision), int(chunk_size), _cout(fs_re, fs_im), _ptr(workspace),
        int(workspace.numel()), ctypes.c_void_p(s.cuda_stream))
    if check and rc != SSDC_OK:
        raise SSDCError(rc, "ssd_complex_final_state")
    return rc


class FinalState:
    """The state a scan leaves (ssd_complex_final_state) with its output and workspace
    held: no allocation per call."""

    def __init__(self, Bn, T, H, N, D, chunk_size, precision="tf32", device="cuda"):
        import torch
        self.shape = (Bn, T, H, N, D)
        self.chunk_size = int(chunk_size)
        self.precision = precision
        d = dims(Bn, T, H, N, D, precision)
        rc = ssd_complex_fwd_supported(d, chunk_size)
        if rc != SSDC_OK:
            raise SSDCError(rc, "ssd_complex_fwd_supported")
        nbytes = load().ssd_complex_final_state_workspace_bytes(d, int(chunk_size))
        self.fs_re = torch.empty((Bn, H, N, D), dtype=torch.float32, device=device)
        self.fs_im = torch.empty((Bn, H, N, D), dtype=torch.float32, device=device)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)

    def __call__(self, x_re, x_im, A_re, A_im, B_re, B_im, dt, stream=None, s0_re=None, s0_im=None):
        ssd_complex_final_state(x_re, x_im, A_re, A_im, B_re, B_im, dt, self.chunk_size, precision=self.precision,
                                s0_re=s0_re, s0_im=s0_im, fs_re=self.fs_re, fs_im=self.fs_im,
                                workspace=self.workspace, stream=stream)
        return self.fs_re, self.fs_im

    def status(self, stream=None) -> int:
        return ssd_complex_status(self.workspace, stream)


def ssd_complex_state_combine(a_re, a_im, s_in_re, s_in_im, s_add_re, s_add_im, *, out_re, out_im,
                              stream=None) -> None:
    """s_out = a s_in + s_add per (b, h); s_in may be (None, None) for zero."""
    import torch
    Bn, H, N, D = s_add_re.shape
    s = torch.cuda.current_stream() if stream is None else stream
    rc = load().ssd_complex_state_combine(_cin(a_re, a_im), _opt_in(s_in_re, s_in_im), _cin(s_add_re, s_add_im),
                                          dims(Bn, 1, H, N, D, "fp32"), _cout(out_re, out_im),
                                          ctypes.c_void_p(s.cuda_stream))
    if rc != SSDC_OK:
        raise SSDCError(rc, "ssd_complex_state_combine")


def ssd_complex_noalloc_status(stream=None) -> int:
    """Device status of the last ssd_complex_fwd_noalloc call (syncs the stream)."""
    import torch

    s = torch.cuda.current_stream() if stream is None else stream
    return load().ssd_complex_noalloc_status(ctypes.c_void_p(s.cuda_stream))


def set_option(option: int, value: int) -> None:
    """Set a process-wide option of the library (ssd_complex_set_option)."""
    rc = load().ssd_complex_set_option(int(option), int(value))
    if rc != SSDC_OK:
        raise SSDCError(rc, "ssd_complex_set_option")


class option:
    """Context manager: set an option for the duration of a block, then restore
    `restore` (the option's default)."""

    DEFAULTS = {OPT_FUSED_CLUSTER: 0, OPT_FUSED_PLANE_MAPS: 1, OPT_TEST_DROP_STATE_CHUNK: -1, OPT_FUSED_KERNEL: 0,
                OPT_MIMO_FUSED: 0}

    def __init__(self, key: int, value: int):
        self.key, self.value = key, value

    def __enter__(self):
        set_option(self.key, self.value)
        return self

    def __exit__(self, *exc):
        set_option(self.key, self.DEFAULTS[self.key])
        return False


def last_launch_count() -> int:
    return load().ssd_complex_last_launch_count()


def last_path() -> str:
    """Name of the path the calling thread's last forward call took (ssd_complex_last_path)."""
    return PATHS.get(load().ssd_complex_last_path(), "none")


def timing_enable(on: bool = True) -> None:
    rc = load().ssd_complex_timing_enable(1 if on else 0)
    if rc != SSDC_OK:
        raise SSDCError(rc, "ssd_complex_timing_enable")


def timing_read(n: int = 8) -> list[float]:
    """Per-launch device times (ms) of the last instrumented forward call."""
    buf = (ctypes.c_float * n)()
    k = load().ssd_complex_timing_read(buf, n)
    if k < 0:
        raise SSDCError(k, "ssd_complex_timing_read")
    return [float(buf[i]) for i in range(min(k, n))]


class Forward:
    """Holds the outputs and the workspace of one problem size, so repeated
    calls allocate nothing. ``__call__`` takes the planar inputs as CUDA
    tensors and returns ``(y_re, y_im, final_state_re, final_state_im)``;
    ``y_re`` is Re(y)."""

    def __init__(self, Bn, T, H, N, D, chunk_size, precision="tf32", device="cuda", bf16_inputs=False):
        """``bf16_inputs``: x, B and C are passed as torch.bfloat16 tensors
        (``ssd_complex_fwd_bf16``; the TF32 precision only)."""
        import torch

        self.shape = (Bn, T, H, N, D)
        self.chunk_size = int(chunk_size)
        self.precision = precision
        self.bf16_inputs = bool(bf16_inputs)
        if self.bf16_inputs and precision != "tf32":
            raise SSDCError(SSDC_ERR_UNSUPPORTED, "bfloat16 inputs run on the TF32 path only")
        d = dims(Bn, T, H, N, D, precision)
        rc = ssd_complex_fwd_supported(d, chunk_size)
        if rc != SSDC_OK:
            raise SSDCError(rc, "ssd_complex_fwd_supported")
        nbytes = ssd_complex_fwd_workspace_bytes(d, chunk_size)
        f32 = dict(dtype=torch.float32, device=device)
        self.y_re = torch.empty((Bn, T, H, D), **f32)
        self.y_im = torch.empty((Bn, T, H, D), **f32)
        self.fs_re = torch.empty((Bn, H, N, D), **f32)
        self.fs_im = torch.empty((Bn, H, N, D), **f32)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)

    def __call__(self, x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt, stream=None,
                 s0_re=None, s0_im=None):
        """``s0_re, s0_im``: an optional initial state (B,H,N,D); passing this
        object's own ``fs_re, fs_im`` continues the previous call in place."""
        if self.bf16_inputs:
            ssd_complex_fwd_bf16(x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt, self.chunk_size,
                                 s0_re=s0_re, s0_im=s0_im, y_re=self.y_re, y_im=self.y_im, fs_re=self.fs_re,
                                 fs_im=self.fs_im, workspace=self.workspace, stream=stream)
        elif s0_re is None and s0_im is None:
            ssd_complex_fwd_ws(x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt, self.chunk_size,
                               precision=self.precision, y_re=self.y_re, y_im=self.y_im,
                               fs_re=self.fs_re, fs_im=self.fs_im, workspace=self.workspace,
                               stream=stream)
        else:
            ssd_complex_fwd_init(x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt, s0_re, s0_im,
                                 self.chunk_size, precision=self.precision, y_re=self.y_re,
                                 y_im=self.y_im, fs_re=self.fs_re, fs_im=self.fs_im,
                                 workspace=self.workspace, stream=stream)
        return self.y_re, self.y_im, self.fs_re, self.fs_im

    def status(self, stream=None) -> int:
        return ssd_complex_status(self.workspace, stream)


def ssd_complex_fwd(x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt, chunk_size, precision="tf32",
                    stream=None):
    """Call ``ssd_complex_fwd`` (workspace allocated stream-ordered by the library) on
    torch CUDA tensors; returns new (y_re, y_im, fs_re, fs_im) tensors. ``x_im`` may be
    None for a real x."""
    import torch

    Bn, T, H, D = x_re.shape
    N = B_re.shape[-1]
    f32 = dict(dtype=torch.float32, device=x_re.device)
    y_re, y_im = torch.empty((Bn, T, H, D), **f32), torch.empty((Bn, T, H, D), **f32)
    fs_re, fs_im = torch.empty((Bn, H, N, D), **f32), torch.empty((Bn, H, N, D), **f32)
    s = torch.cuda.current_stream() if stream is None else stream
    rc = load().ssd_complex_fwd(
        _cin(x_re, x_im), _cin(A_re, A_im), _cin(B_re, B_im), _cin(C_re, C_im), _ptr(dt),
        dims(Bn, T, H, N, D, precision), int(chunk_size), _cout(y_re, y_im), _cout(fs_re, fs_im),
        ctypes.c_void_p(s.cuda_stream))
    if rc != SSDC_OK:
        raise SSDCError(rc, "ssd_complex_fwd")
    return y_re, y_im, fs_re, fs_im


class HostForward:
    """The host-buffer form of ``Forward``: holds pinned host outputs and the
    device scratch of one problem size. ``__call__`` takes the planar inputs as
    contiguous float32 CPU tensors (pinned for overlapped copies) and returns
    ``(y_re, y_im, final_state_re, final_state_im)`` as CPU tensors, filled
    when the call returns."""

    def __init__(self, Bn, T, H, N, D, chunk_size, precision="tf32", device="cuda"):
        import torch

        self.shape = (Bn, T, H, N, D)
        self.chunk_size = int(chunk_size)
        self.precision = precision
        d = dims(Bn, T, H, N, D, precision)
        rc = ssd_complex_fwd_supported(d, chunk_size)
        if rc != SSDC_OK:
            raise SSDCError(rc, "ssd_complex_fwd_supported")
        pin = torch.cuda.is_available()
        f32 = dict(dtype=torch.float32, pin_memory=pin)
        self.y_re = torch.empty((Bn, T, H, D), **f32)
        self.y_im = torch.empty((Bn, T, H, D), **f32)
        self.fs_re = torch.empty((Bn, H, N, D), **f32)
        self.fs_im = torch.empty((Bn, H, N, D), **f32)
        nbytes = ssd_complex_fwd_host_scratch_bytes(d, chunk_size)
        self.scratch = torch.empty(nbytes, dtype=torch.uint8, device=device)

    def __call__(self, x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt, stream=None):
        ssd_complex_fwd_host(x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt, self.chunk_size,
                             precision=self.precision, y_re=self.y_re, y_im=self.y_im,
                             fs_re=self.fs_re, fs_im=self.fs_im, scratch=self.scratch,
                             stream=stream)
        return self.y_re, self.y_im, self.fs_re, self.fs_im
