"""Python binding of libssmscan.so: argument marshalling only.

Every step of the scan runs in the library's CUDA kernels; this module checks tensor
placement and dtypes, fills the C params structs declared in include/ssmscan.h, allocates
outputs and workspace with PyTorch (which owns device memory and streams) and calls the
C ABI on the current torch stream. There is no CPU or PyTorch fallback: if the library is
missing or a call fails, an exception says why.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# SSMSCAN_LIBRARY selects another build of the library (e.g. the index-checking
# libssmscan_debug.so): a path, or a file name in the package directory.
LIB_PATH = os.path.join(_PKG, os.environ.get("SSMSCAN_LIBRARY", "libssmscan.so"))

SSM_OK, SSM_ERR_INVALID_ARG, SSM_ERR_UNSUPPORTED, SSM_ERR_CUDA, SSM_ERR_TIMEOUT, SSM_ERR_WORKSPACE, SSM_ERR_BOUNDS = \
    range(7)
SSM_DTYPE_F32, SSM_DTYPE_BF16 = 0, 1
SSM_DISC_DELTA_B, SSM_DISC_ZOH = 0, 1
ABI_VERSION = 4
WORKSPACE_HEADER_BYTES = 256   # SSM_WORKSPACE_HEADER_BYTES: the status word of a workspace

# Every function the header declares (checked by the CPU test suite).
EXPORTS = ("ssm_scan_workspace_size", "ssm_scan_fwd", "ssd_chunk_scan_workspace_size", "ssd_chunk_scan_fwd",
           "ssm_check_status", "ssm_status_string", "ssm_last_error", "ssm_abi_version",
           "ssm_kernel_launch_count", "ssm_scan_fwd_noalloc", "ssm_noalloc_scratch_bytes",
           "ssm_causal_conv1d_workspace_size", "ssm_causal_conv1d_fwd")

_i64, _i32, _vp, _sz = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t


class ScanParams(ctypes.Structure):
    _fields_ = [("batch", _i64), ("seqlen", _i64), ("dim", _i64), ("dstate", _i64),
                ("io_dtype", _i32), ("delta_softplus", _i32), ("reverse", _i32), ("discretization", _i32),
                ("x", _vp), ("delta", _vp), ("B", _vp), ("C", _vp), ("z", _vp),
                ("A", _vp), ("D", _vp), ("delta_bias", _vp), ("h0", _vp), ("y", _vp), ("h_last", _vp),
                ("x_stride", _i64 * 3), ("delta_stride", _i64 * 3), ("z_stride", _i64 * 3),
                ("y_stride", _i64 * 3), ("B_stride", _i64 * 3), ("C_stride", _i64 * 3),
                ("chunk_len", _i64), ("workspace", _vp), ("workspace_bytes", _sz),
                ("debug_flags", _i32), ("reserved", _i32),
                ("conv_weight", _vp), ("conv_bias", _vp), ("conv_x_prev", _vp), ("conv_width", _i32),
                ("reserved2", _i32), ("phase_events", ctypes.POINTER(_vp)), ("n_phase_events", _i32),
                ("algorithm", _i32)]


class Conv1dParams(ctypes.Structure):
    _fields_ = [("batch", _i64), ("seqlen", _i64), ("dim", _i64), ("width", _i32), ("io_dtype", _i32),
                ("silu", _i32), ("reserved", _i32), ("x", _vp), ("weight", _vp), ("bias", _vp),
                ("x_prev", _vp), ("y", _vp), ("workspace", _vp), ("workspace_bytes", _sz)]

SSM_DEBUG_SKIP_FIRST_LOAD = 1


class SSDParams(ctypes.Structure):
    _fields_ = [("batch", _i64), ("seqlen", _i64), ("nheads", _i64), ("headdim", _i64), ("dstate", _i64),
                ("ngroups", _i64), ("chunk_size", _i64), ("io_dtype", _i32), ("delta_softplus", _i32),
                ("x", _vp), ("delta", _vp), ("A", _vp), ("B", _vp), ("C", _vp), ("D", _vp), ("z", _vp),
                ("delta_bias", _vp), ("h0", _vp), ("y", _vp), ("h_last", _vp),
                ("workspace", _vp), ("workspace_bytes", _sz)]


class SSMError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{_status_name(status)}: {message}")


_lib = None
_lock = threading.Lock()


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libssmscan.so (built in-tree by ``python -m selective_state_space_127_b300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: build it with "
                                   "`python -m selective_state_space_127_b300.build` (there is no fallback)")
            lib = ctypes.CDLL(path)
            lib.ssm_scan_workspace_size.argtypes = [ctypes.POINTER(ScanParams)]
            lib.ssm_scan_workspace_size.restype = _sz
            lib.ssm_scan_fwd.argtypes = [ctypes.POINTER(ScanParams), _vp]
            lib.ssm_scan_fwd.restype = ctypes.c_int
            lib.ssd_chunk_scan_workspace_size.argtypes = [ctypes.POINTER(SSDParams)]
            lib.ssd_chunk_scan_workspace_size.restype = _sz
            lib.ssd_chunk_scan_fwd.argtypes = [ctypes.POINTER(SSDParams), _vp]
            lib.ssd_chunk_scan_fwd.restype = ctypes.c_int
            lib.ssm_check_status.argtypes = [_vp, _vp, ctypes.c_int]
            lib.ssm_check_status.restype = ctypes.c_int
            lib.ssm_noalloc_scratch_bytes.argtypes = []
            lib.ssm_noalloc_scratch_bytes.restype = _sz
            lib.ssm_causal_conv1d_workspace_size.argtypes = [ctypes.POINTER(Conv1dParams)]
            lib.ssm_causal_conv1d_workspace_size.restype = _sz
            lib.ssm_status_string.argtypes = [ctypes.c_int]
            lib.ssm_status_string.restype = ctypes.c_char_p
            lib.ssm_last_error.argtypes = []
            lib.ssm_last_error.restype = ctypes.c_char_p
            lib.ssm_abi_version.argtypes = []
            lib.ssm_abi_version.restype = ctypes.c_int
            lib.ssm_scan_fwd_noalloc.argtypes = [ctypes.POINTER(ScanParams), _vp]
            lib.ssm_scan_fwd_noalloc.restype = ctypes.c_int
            lib.ssm_causal_conv1d_fwd.argtypes = [ctypes.POINTER(Conv1dParams), _vp]
            lib.ssm_causal_conv1d_fwd.restype = ctypes.c_int
            lib.ssm_kernel_launch_count.argtypes = []
            lib.ssm_kernel_launch_count.restype = ctypes.c_uint64
            if lib.ssm_abi_version() != ABI_VERSION:
                raise RuntimeError(f"{path}: ABI version {lib.ssm_abi_version()} != {ABI_VERSION}")
            _lib = lib
    return _lib


def _status_name(s: int) -> str:
    return ["SSM_OK", "SSM_ERR_INVALID_ARG", "SSM_ERR_UNSUPPORTED", "SSM_ERR_CUDA", "SSM_ERR_TIMEOUT",
            "SSM_ERR_WORKSPACE", "SSM_ERR_BOUNDS"][s] if 0 <= s <= 6 else f"status {s}"


def _check(lib, status: int):
    if status != SSM_OK:
        raise SSMError(status, lib.ssm_last_error().decode(errors="replace"))


def _io_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SSM_DTYPE_F32
    if t.dtype == torch.bfloat16:
        return SSM_DTYPE_BF16
    raise TypeError(f"I/O tensors must be float32 or bfloat16, got {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _strides3(t, n_expected_dims=3):
    if t is None:
        return (0, 0, 0)
    if t.dim() != n_expected_dims:
        raise ValueError(f"expected a {n_expected_dims}-d tensor, got shape {tuple(t.shape)}")
    return tuple(int(s) for s in t.stride())


def _f32_contig(name, t, shape, device):
    if t is None:
        return None
    if t.dtype != torch.float32 or not t.is_contiguous() or tuple(t.shape) != tuple(shape) or t.device != device:
        raise ValueError(f"{name} must be a contiguous float32 tensor of shape {tuple(shape)} on {device}")
    return t


def _stream_handle(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def new_workspace(nbytes: int, device) -> torch.Tensor:
    """A device workspace of ``nbytes`` (at least the status header) with its header zeroed, as
    the library expects before a workspace's first use. PyTorch's allocator returns blocks
    aligned to at least 256 bytes."""
    return torch.zeros(max(int(nbytes), WORKSPACE_HEADER_BYTES), dtype=torch.uint8, device=device)


def noalloc_scratch_bytes() -> int:
    """Size of the built-in scratch of ssm_scan_fwd_noalloc, as compiled into the library."""
    return int(load_library().ssm_noalloc_scratch_bytes())


def _event_array(events):
    """ctypes array of cudaEvent_t handles of torch.cuda.Event objects (each created by a
    record on the current stream first, since torch creates events lazily)."""
    if not events:
        return None, 0
    handles = []
    for ev in events:
        if ev.cuda_event == 0:
            ev.record()
        handles.append(ev.cuda_event)
    arr = (_vp * len(handles))(*handles)
    return arr, len(handles)


# ssm_scan_params.algorithm: the serial walk (default) or the in-tile associative scan
SSM_SCAN_ALGO_SERIAL, SSM_SCAN_ALGO_ASSOC = 0, 1
_ALGOS = {"serial": SSM_SCAN_ALGO_SERIAL, "assoc": SSM_SCAN_ALGO_ASSOC}


def _scan_params(x, delta, A, B, C, D=None, z=None, delta_bias=None, *, delta_softplus=True, h0=None,
                 reverse=False, zoh=False, chunk_len=0, out=None, return_last_state=True, h_last=None,
                 debug_flags=0, conv_weight=None, conv_bias=None, conv_x_prev=None, phase_events=None,
                 algorithm="serial"):
    """Check the tensors and fill a ScanParams; returns (params, y, h_last)."""
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor (use ssm_scan_fwd_host for host buffers)")
    dev = x.device
    b, L, Dm = x.shape
    N = A.shape[1]
    io = _io_dtype(x)
    for name, t, shp in (("delta", delta, (b, L, Dm)), ("B", B, (b, L, N)), ("C", C, (b, L, N)),
                         ("z", z, (b, L, Dm))):
        if t is None:
            continue
        if t.device != dev or t.dtype != x.dtype or tuple(t.shape) != shp:
            raise ValueError(f"{name} must be {x.dtype} of shape {shp} on {dev}, got {t.dtype} "
                             f"{tuple(t.shape)} on {t.device}")
    _f32_contig("A", A, (Dm, N), dev)
    _f32_contig("D", D, (Dm,), dev)
    _f32_contig("delta_bias", delta_bias, (Dm,), dev)
    _f32_contig("h0", h0, (b, Dm, N), dev)
    K = 0
    if conv_weight is not None:
        K = conv_weight.shape[-1]
        _f32_contig("conv_weight", conv_weight, (Dm, K), dev)
        _f32_contig("conv_bias", conv_bias, (Dm,), dev)
        if conv_x_prev is not None and (conv_x_prev.dtype != x.dtype or tuple(conv_x_prev.shape) != (b, K - 1, Dm)
                                        or not conv_x_prev.is_contiguous() or conv_x_prev.device != dev):
            raise ValueError(f"conv_x_prev must be contiguous {x.dtype} of shape {(b, K - 1, Dm)} on {dev}")
    y = out if out is not None else torch.empty((b, L, Dm), device=dev, dtype=x.dtype)
    if y.dtype != x.dtype or tuple(y.shape) != (b, L, Dm) or y.device != dev:
        raise ValueError("out has the wrong dtype, shape or device")
    hl = h_last
    if hl is None and return_last_state:
        hl = torch.empty((b, Dm, N), device=dev, dtype=torch.float32)
    _f32_contig("h_last", hl, (b, Dm, N), dev)
    p = ScanParams()
    p.batch, p.seqlen, p.dim, p.dstate = b, L, Dm, N
    p.io_dtype, p.delta_softplus, p.reverse = io, int(bool(delta_softplus)), int(bool(reverse))
    p.discretization = SSM_DISC_ZOH if zoh else SSM_DISC_DELTA_B
    p.x, p.delta, p.B, p.C, p.z = _ptr(x), _ptr(delta), _ptr(B), _ptr(C), _ptr(z)
    p.A, p.D, p.delta_bias, p.h0 = _ptr(A), _ptr(D), _ptr(delta_bias), _ptr(h0)
    p.y, p.h_last = _ptr(y), _ptr(hl)
    p.x_stride[:] = _strides3(x)
    p.delta_stride[:] = _strides3(delta)
    p.z_stride[:] = _strides3(z)
    p.y_stride[:] = _strides3(y)
    p.B_stride[:] = _strides3(B)
    p.C_stride[:] = _strides3(C)
    p.chunk_len = int(chunk_len)
    p.debug_flags = int(debug_flags)
    if algorithm not in _ALGOS:
        raise ValueError(f"algorithm must be one of {sorted(_ALGOS)}")
    p.algorithm = _ALGOS[algorithm]
    if conv_weight is not None:
        p.conv_weight, p.conv_bias, p.conv_x_prev = _ptr(conv_weight), _ptr(conv_bias), _ptr(conv_x_prev)
        p.conv_width = K
    arr, n = _event_array(phase_events)
    if arr is not None:
        p.phase_events, p.n_phase_events = ctypes.cast(arr, ctypes.POINTER(_vp)), n
        p._events_keepalive = arr
    return p, y, hl


def scan_workspace_size(x, delta, A, B, C, D=None, z=None, delta_bias=None, **kw) -> int:
    """Bytes of device workspace ssm_scan_fwd needs for these arguments (0 if none)."""
    lib = load_library()
    kw = {k: v for k, v in kw.items() if k not in ("stream", "workspace")}
    p, _, _ = _scan_params(x, delta, A, B, C, D, z, delta_bias, **kw)
    n = lib.ssm_scan_workspace_size(ctypes.byref(p))
    if n == ctypes.c_size_t(-1).value:
        _check(lib, lib.ssm_scan_fwd(ctypes.byref(p), None))  # raises with the reason
    return int(n)


def ssm_scan_fwd(x, delta, A, B, C, D=None, z=None, delta_bias=None, *, delta_softplus=True, h0=None,
                 reverse=False, zoh=False, chunk_len=0, out=None, return_last_state=True, h_last=None,
                 stream=None, workspace=None, debug_flags=0, conv_weight=None, conv_bias=None, conv_x_prev=None,
                 phase_events=None, algorithm="serial"):
    """Selective scan on the GPU. x, delta, z: (b, L, D); B, C: (b, L, N); A: (D, N) fp32;
    D, delta_bias: (D) fp32; h0: (b, D, N) fp32. I/O tensors are fp32 or bf16 (all alike) and
    may be strided (delta's channel stride may be 0). ``workspace`` (a uint8 CUDA tensor of at
    least scan_workspace_size() bytes, 256-byte aligned, its first 256 bytes zeroed before
    first use, e.g. from new_workspace()) holds the status word read by check_status() and the
    chunk carries of long sequences; a fresh one is allocated when not given (or too small).
    With ``conv_weight`` (D, K) fp32 (K <= 4), x is the raw input and the scan runs on
    silu(causal conv1d(x) + conv_bias); ``conv_x_prev`` (b, K-1, D) holds the K-1 raw inputs
    before x[:, 0] (zeros when None). ``phase_events``: torch.cuda.Event objects recorded
    before the call's first kernel and after each kernel. ``algorithm``: "serial" (default:
    each lane walks its states' steps) or "assoc" (an in-tile associative scan of the
    (A_bar, B_bar x) pairs over a warp's lanes; N = 16 or 32, forward, delta B, TMA layout).
    Returns (y, h_last or None)."""
    lib = load_library()
    p, y, hl = _scan_params(x, delta, A, B, C, D, z, delta_bias, delta_softplus=delta_softplus, h0=h0,
                            reverse=reverse, zoh=zoh, chunk_len=chunk_len, out=out,
                            return_last_state=return_last_state, h_last=h_last, debug_flags=debug_flags,
                            conv_weight=conv_weight, conv_bias=conv_bias, conv_x_prev=conv_x_prev,
                            phase_events=phase_events, algorithm=algorithm)
    ws_bytes = lib.ssm_scan_workspace_size(ctypes.byref(p))
    if ws_bytes == ctypes.c_size_t(-1).value:
        _check(lib, lib.ssm_scan_fwd(ctypes.byref(p), None))  # raises with the reason
    if ws_bytes > 0:
        ws = workspace
        if ws is None or ws.numel() < ws_bytes:
            ws = new_workspace(ws_bytes, x.device)
        p.workspace, p.workspace_bytes = _ptr(ws), ws.numel()
    with torch.cuda.device(x.device):
        _check(lib, lib.ssm_scan_fwd(ctypes.byref(p), _stream_handle(stream)))
    return y, hl


class ScanCall:
    """A prepared selective-scan call for repeated use on the same buffers (a decode loop, a
    benchmark): the arguments of ssm_scan_fwd are checked and the C params struct is filled
    once, with the outputs and the workspace bound; each call then only enqueues the C call on
    the stream. Returns (y, h_last) like ssm_scan_fwd."""

    def __init__(self, x, delta, A, B, C, D=None, z=None, delta_bias=None, *, out=None, h_last=None,
                 workspace=None, stream=None, **kw):
        self._lib = load_library()
        p, self.y, self.h_last = _scan_params(x, delta, A, B, C, D, z, delta_bias, out=out, h_last=h_last, **kw)
        n = self._lib.ssm_scan_workspace_size(ctypes.byref(p))
        if n == ctypes.c_size_t(-1).value:
            _check(self._lib, self._lib.ssm_scan_fwd(ctypes.byref(p), None))
        self.workspace = workspace if workspace is not None and workspace.numel() >= n else \
            (new_workspace(n, x.device) if n > 0 else None)
        if self.workspace is not None:
            p.workspace, p.workspace_bytes = _ptr(self.workspace), self.workspace.numel()
        self._p = p
        self._ref = ctypes.byref(p)
        self._device = x.device
        self._keep = (x, delta, A, B, C, D, z, delta_bias, kw.get("h0"), kw.get("conv_weight"),
                      kw.get("conv_bias"), kw.get("conv_x_prev"))
        self._stream = _stream_handle(stream) if stream is not None else None

    def __call__(self, stream=None):
        if stream is not None:
            sh = _stream_handle(stream)
        elif self._stream is not None:
            sh = self._stream
        else:
            sh = ctypes.c_void_p(torch.cuda.current_stream(self._device).cuda_stream)
        s = self._lib.ssm_scan_fwd(self._ref, sh)
        if s != SSM_OK:
            _check(self._lib, s)
        return self.y, self.h_last


def ssm_scan_fwd_noalloc(x, delta, A, B, C, D=None, z=None, delta_bias=None, *, delta_softplus=True, h0=None,
                         chunk_len=0, out=None, return_last_state=True, h_last=None, stream=None):
    """The allocation-free C entry point (no workspace: the library's built-in scratch is
    used; its status word is read by check_status(None)). Outputs are allocated here when not
    given; pass ``out`` and ``h_last`` to keep the call itself free of allocations. Returns
    (y, h_last or None)."""
    lib = load_library()
    p, y, hl = _scan_params(x, delta, A, B, C, D, z, delta_bias, delta_softplus=delta_softplus, h0=h0,
                            chunk_len=chunk_len, out=out, return_last_state=return_last_state, h_last=h_last)
    with torch.cuda.device(x.device):
        _check(lib, lib.ssm_scan_fwd_noalloc(ctypes.byref(p), _stream_handle(stream)))
    return y, hl


def causal_conv1d_fwd(x, weight, bias=None, *, silu=True, x_prev=None, out=None, stream=None, workspace=None):
    """Causal depthwise conv1d along t (then SiLU when ``silu``) on the GPU. x: (b, L, D)
    contiguous fp32 or bf16 with D * element size a multiple of 16 bytes; weight: (D, K) fp32
    (K <= 4; weight[:, K-1] multiplies x_t); bias: (D) fp32; x_prev: (b, K-1, D) like x, the
    inputs before x[:, 0] (zeros when None). Returns y (b, L, D) in x's dtype."""
    lib = load_library()
    if not x.is_cuda or not x.is_contiguous() or x.dim() != 3:
        raise ValueError("x must be a contiguous (b, L, D) CUDA tensor")
    dev = x.device
    b, L, Dm = x.shape
    K = weight.shape[-1]
    _f32_contig("weight", weight, (Dm, K), dev)
    _f32_contig("bias", bias, (Dm,), dev)
    if x_prev is not None and (x_prev.dtype != x.dtype or tuple(x_prev.shape) != (b, K - 1, Dm)
                               or not x_prev.is_contiguous() or x_prev.device != dev):
        raise ValueError(f"x_prev must be contiguous {x.dtype} of shape {(b, K - 1, Dm)} on {dev}")
    y = out if out is not None else torch.empty_like(x)
    if y.dtype != x.dtype or tuple(y.shape) != (b, L, Dm) or not y.is_contiguous() or y.device != dev:
        raise ValueError("out has the wrong dtype, shape, layout or device")
    p = Conv1dParams()
    p.batch, p.seqlen, p.dim, p.width = b, L, Dm, K
    p.io_dtype, p.silu = _io_dtype(x), int(bool(silu))
    p.x, p.weight, p.bias, p.x_prev, p.y = _ptr(x), _ptr(weight), _ptr(bias), _ptr(x_prev), _ptr(y)
    ws_bytes = lib.ssm_causal_conv1d_workspace_size(ctypes.byref(p))
    if ws_bytes == ctypes.c_size_t(-1).value:
        _check(lib, lib.ssm_causal_conv1d_fwd(ctypes.byref(p), None))
    if ws_bytes > 0:
        ws = workspace if workspace is not None and workspace.numel() >= ws_bytes else new_workspace(ws_bytes, dev)
        p.workspace, p.workspace_bytes = _ptr(ws), ws.numel()
    with torch.cuda.device(dev):
        _check(lib, lib.ssm_causal_conv1d_fwd(ctypes.byref(p), _stream_handle(stream)))
    return y


def ssd_chunk_scan_fwd(x, delta, A, B, C, chunk_size=256, D=None, z=None, delta_bias=None, *,
                       delta_softplus=True, h0=None, out=None, return_last_state=True, h_last=None,
                       stream=None, workspace=None):
    """SSD chunked scan on the GPU. x, z: (b, L, H, P); delta: (b, L, H); A, D, delta_bias: (H)
    fp32; B, C: (b, L, G, N) or (b, L, N); h0: (b, H, N, P) fp32. Contiguous tensors only.
    Returns (y, h_last or None)."""
    lib = load_library()
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    dev = x.device
    if B.dim() == 3:
        B, C = B.unsqueeze(2), C.unsqueeze(2)
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    io = _io_dtype(x)
    for name, t, shp in (("x", x, (b, L, H, P)), ("delta", delta, (b, L, H)), ("B", B, (b, L, G, N)),
                         ("C", C, (b, L, G, N)), ("z", z, (b, L, H, P))):
        if t is None:
            continue
        if t.device != dev or t.dtype != x.dtype or tuple(t.shape) != shp or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {x.dtype} tensor of shape {shp} on {dev}")
    _f32_contig("A", A, (H,), dev)
    _f32_contig("D", D, (H,), dev)
    _f32_contig("delta_bias", delta_bias, (H,), dev)
    _f32_contig("h0", h0, (b, H, N, P), dev)
    y = out if out is not None else torch.empty((b, L, H, P), device=dev, dtype=x.dtype)
    hl = h_last
    if hl is None and return_last_state:
        hl = torch.empty((b, H, N, P), device=dev, dtype=torch.float32)
    _f32_contig("h_last", hl, (b, H, N, P), dev)
    p = SSDParams()
    p.batch, p.seqlen, p.nheads, p.headdim, p.dstate, p.ngroups = b, L, H, P, N, G
    p.chunk_size, p.io_dtype, p.delta_softplus = int(chunk_size), io, int(bool(delta_softplus))
    p.x, p.delta, p.A, p.B, p.C, p.D, p.z = _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z)
    p.delta_bias, p.h0, p.y, p.h_last = _ptr(delta_bias), _ptr(h0), _ptr(y), _ptr(hl)
    ws_bytes = lib.ssd_chunk_scan_workspace_size(ctypes.byref(p))
    if ws_bytes == ctypes.c_size_t(-1).value:
        _check(lib, lib.ssd_chunk_scan_fwd(ctypes.byref(p), None))
    if ws_bytes > 0:
        ws = workspace if workspace is not None and workspace.numel() >= ws_bytes else new_workspace(ws_bytes, dev)
        p.workspace, p.workspace_bytes = _ptr(ws), ws.numel()
    with torch.cuda.device(dev):
        _check(lib, lib.ssd_chunk_scan_fwd(ctypes.byref(p), _stream_handle(stream)))
    return y, hl


_PER_ROW = ("x", "delta", "z", "B", "C")


def ssm_scan_fwd_host(inputs: dict, device="cuda", stream=None, dev_buffers: dict | None = None, slices=None,
                      segments=None, **kw):
    """End-to-end call for pinned host buffers: copy the inputs to the device, run
    ssm_scan_fwd, copy y and h_last back into pinned host tensors, synchronise.

    The work is cut into pieces whose host-to-device copy, scan and device-to-host copy run on
    three streams (copy in, compute, copy out), so that the copies of one piece overlap the scan
    and the copies of its neighbours. With at least ``slices`` (default 4) batch rows the pieces
    are groups of rows, which are independent. With fewer rows the pieces are ``segments``
    (default 8) stretches of the sequence, scanned in order: each stretch starts from the state
    the previous one left in the device copy of h_last (the call reads h0 before it writes
    h_last, so the two may be one buffer), and with the conv prologue it takes the K-1 raw inputs
    before it from the device copy of x. ``dev_buffers`` (a dict) keeps the device tensors, the
    pinned outputs and the streams between calls. Returns (y_host, h_last_host)."""
    dev = torch.device(device)
    cache = dev_buffers if dev_buffers is not None else {}
    x = inputs["x"]
    b, L = x.shape[0], x.shape[1]
    nsl = slices or 4
    if b >= nsl or L == 0:
        rows = [(i * b // nsl, (i + 1) * b // nsl) for i in range(min(b, nsl))] or [(0, b)]
        pieces = [((r0, r1), (0, L)) for r0, r1 in rows]
    else:
        nseg = max(1, min(segments or 8, L // 64))
        cuts = [((i * L // nseg) // 64) * 64 for i in range(nseg)] + [L]   # 64-step aligned starts
        segs = [(cuts[i], cuts[i + 1]) for i in range(nseg) if cuts[i + 1] > cuts[i]]
        if kw.get("reverse"):
            segs = segs[::-1]
        pieces = [((0, b), sg) for sg in segs]
    if "_streams" not in cache:
        cache["_streams"] = tuple(torch.cuda.Stream(device=dev) for _ in range(3))
    s_in, s_comp, s_out = cache["_streams"]
    caller = stream if stream is not None else torch.cuda.current_stream(dev)
    s_in.wait_stream(caller)

    def dev_buf(name, like):
        t = cache.get(name)
        if t is None or t.shape != like.shape or t.dtype != like.dtype:
            t = torch.empty(like.shape, dtype=like.dtype, device=dev)
            cache[name] = t
        return t

    d = {k: (dev_buf(k, v) if v is not None else None) for k, v in inputs.items()}
    N = inputs["A"].shape[1]
    y_dev = dev_buf("_y", x)
    hl_dev = dev_buf("_h_last", torch.empty((b, x.shape[2], N), dtype=torch.float32, device="meta"))
    y_host = cache.get("_y_host")
    if y_host is None or y_host.shape != x.shape or y_host.dtype != x.dtype:
        y_host = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
        cache["_y_host"] = y_host
    hl_host = cache.get("_h_last_host")
    if hl_host is None or hl_host.shape != hl_dev.shape:
        hl_host = torch.empty(hl_dev.shape, dtype=torch.float32, pin_memory=True)
        cache["_h_last_host"] = hl_host
    seq_split = len(pieces) > 1 and pieces[0][0] == (0, b)
    with torch.cuda.stream(s_in):
        for k, v in inputs.items():        # per-channel inputs and h0: all at once
            if v is not None and (k not in _PER_ROW + ("h0",) or (k == "h0" and seq_split)):
                d[k].copy_(v, non_blocking=True)
    ckw = {k: v for k, v in kw.items() if k not in ("workspace", "conv_x_prev")}
    conv_w = d["conv_weight"] if d.get("conv_weight") is not None else kw.get("conv_weight")
    xprev0 = d["conv_x_prev"] if d.get("conv_x_prev") is not None else kw.get("conv_x_prev")
    for i, ((r0, r1), (s0, s1)) in enumerate(pieces):
        with torch.cuda.stream(s_in):
            for k in _PER_ROW:
                if inputs.get(k) is None:
                    continue
                if s0 == 0 and s1 == L:
                    d[k][r0:r1].copy_(inputs[k][r0:r1], non_blocking=True)
                else:                       # one contiguous stretch per row
                    for r in range(r0, r1):
                        d[k][r, s0:s1].copy_(inputs[k][r, s0:s1], non_blocking=True)
            if not seq_split and inputs.get("h0") is not None:
                d["h0"][r0:r1].copy_(inputs["h0"][r0:r1], non_blocking=True)
        s_comp.wait_stream(s_in)
        sl = {k: (v[r0:r1, s0:s1] if k in _PER_ROW else v) for k, v in d.items() if k not in ("h0", "conv_x_prev")}
        if seq_split:
            h0 = (d["h0"] if d.get("h0") is not None else None) if i == 0 else hl_dev
        else:
            h0 = d["h0"][r0:r1] if d.get("h0") is not None else None
        xprev = xprev0[r0:r1] if xprev0 is not None else None
        if conv_w is not None and s0 > 0:   # the raw inputs before this stretch are on the device
            K = conv_w.shape[-1]
            with torch.cuda.stream(s_comp):
                xprev = d["x"][r0:r1, s0 - (K - 1):s0].contiguous()
        need = scan_workspace_size(**sl, h0=h0, **ckw)
        ws = cache.get("_workspace")
        if need > 0 and (ws is None or ws.numel() < need):
            with torch.cuda.stream(s_comp):
                ws = new_workspace(need, dev)
            cache["_workspace"] = ws
        ssm_scan_fwd(**sl, h0=h0, out=y_dev[r0:r1, s0:s1], h_last=hl_dev[r0:r1], stream=s_comp,
                     workspace=ws if need > 0 else None, conv_x_prev=xprev, **ckw)
        s_out.wait_stream(s_comp)
        with torch.cuda.stream(s_out):
            if s0 == 0 and s1 == L:
                y_host[r0:r1].copy_(y_dev[r0:r1], non_blocking=True)
            else:
                for r in range(r0, r1):
                    y_host[r, s0:s1].copy_(y_dev[r, s0:s1], non_blocking=True)
            if not seq_split:
                hl_host[r0:r1].copy_(hl_dev[r0:r1], non_blocking=True)
    if seq_split:
        with torch.cuda.stream(s_out):
            hl_host.copy_(hl_dev, non_blocking=True)
    s_out.synchronize()
    return y_host, hl_host


def kernel_launch_count() -> int:
    """Kernels the library has enqueued in this process so far."""
    return int(load_library().ssm_kernel_launch_count())


def check_status(workspace, clear: bool = True, stream=None) -> int:
    """Synchronise the stream and return the status word of ``workspace`` (the uint8 tensor
    given to earlier calls; None = the built-in scratch of ssm_scan_fwd_noalloc): SSM_OK or
    SSM_ERR_TIMEOUT. Clears it by default."""
    lib = load_library()
    ptr = None if workspace is None else ctypes.c_void_p(workspace.data_ptr())
    return lib.ssm_check_status(ptr, _stream_handle(stream), int(bool(clear)))
