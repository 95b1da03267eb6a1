"""ctypes binding of libssd (include/ssd.h): argument marshalling only.

Every function here has the name of the C entry point it forwards to.  Tensors
are torch tensors on the CUDA device (contiguous, 16-byte aligned); the stream
defaults to torch's current stream.  Errors come back as SsdError carrying the
library's status.  Nothing here computes any part of the layer: if libssd.so
is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Sequence

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libssd.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "ssd.h")

SSD_OK, SSD_ERR_INVALID_ARG, SSD_ERR_UNSUPPORTED, SSD_ERR_CUDA, SSD_ERR_TIMEOUT = range(5)
SSD_F32, SSD_BF16 = 0, 1


class SsdError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, ssd_status_string(status), status))


class ssd_dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("nheads", ctypes.c_int64),
                ("headdim", ctypes.c_int64), ("dstate", ctypes.c_int64),
                ("ngroups_b", ctypes.c_int64), ("ngroups_c", ctypes.c_int64),
                ("io_dtype", ctypes.c_int32), ("dt_softplus", ctypes.c_int32)]


if not os.path.exists(LIB_PATH):
    raise ImportError("libssd.so is not built (%s); run `python -m state_space_model_09_b300.build`"
                      % LIB_PATH)
_lib = ctypes.CDLL(LIB_PATH)

_vp = ctypes.c_void_p
_P = ctypes.POINTER(ssd_dims)
_lib.ssd_fwd_workspace_size.argtypes = [_P, ctypes.c_int32]
_lib.ssd_fwd_workspace_size.restype = ctypes.c_size_t
_lib.ssd_verify.argtypes = [_P, ctypes.c_int32] + [ctypes.c_void_p] * 14
_lib.ssd_verify.restype = ctypes.c_int32
_lib.ssd_fwd_sequential_workspace_size.argtypes = [_P, ctypes.c_int32, ctypes.c_int64]
_lib.ssd_fwd_sequential_workspace_size.restype = ctypes.c_size_t
_lib.ssd_fwd_sequential.argtypes = [_P] + [ctypes.c_void_p] * 7 + [ctypes.c_int32, ctypes.c_int64] + \
    [ctypes.c_void_p] * 3 + [ctypes.c_size_t, ctypes.c_void_p]
_lib.ssd_fwd_sequential.restype = ctypes.c_int32
_lib.ssd_fwd_num_stages.argtypes = [_P, ctypes.c_int32]
_lib.ssd_fwd_num_stages.restype = ctypes.c_int32
_lib.ssd_fwd_stage_name.argtypes = [_P, ctypes.c_int32, ctypes.c_int32]
_lib.ssd_fwd_stage_name.restype = ctypes.c_char_p
_fwd_args = [_P] + [_vp] * 7 + [ctypes.c_int32, _vp, _vp, _vp, ctypes.c_size_t]
_lib.ssd_fwd.argtypes = _fwd_args + [_vp]
_lib.ssd_fwd.restype = ctypes.c_int
_lib.ssd_fwd_profiled.argtypes = _fwd_args + [_vp, _vp]
_lib.ssd_fwd_profiled.restype = ctypes.c_int
_lib.ssd_fwd_noalloc.argtypes = [_P] + [_vp] * 7 + [ctypes.c_int32, _vp, _vp, _vp]
_lib.ssd_fwd_noalloc.restype = ctypes.c_int
_lib.ssd_multistep.argtypes = [_P] + [_vp] * 11 + [_vp]
_lib.ssd_multistep.restype = ctypes.c_int
_lib.ssd_check_device_error.argtypes = [_vp]
_lib.ssd_check_device_error.restype = ctypes.c_int
_lib.ssd_cp_workspace_size.argtypes = [_P]
_lib.ssd_cp_workspace_size.restype = ctypes.c_size_t
_lib.ssd_cp_segment_decay.argtypes = [_P, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
_lib.ssd_cp_segment_decay.restype = ctypes.c_int
_lib.ssd_cp_correct.argtypes = [_P, ctypes.c_int32, ctypes.c_int32] + [_vp] * 8 + \
    [ctypes.c_size_t, _vp]
_lib.ssd_cp_correct.restype = ctypes.c_int
_lib.ssd_selftest_timeout.argtypes = [ctypes.c_int64, _vp]
_lib.ssd_selftest_timeout.restype = ctypes.c_int
_lib.ssd_status_string.argtypes = [ctypes.c_int]
_lib.ssd_status_string.restype = ctypes.c_char_p
_lib.ssd_version.argtypes = []
_lib.ssd_version.restype = ctypes.c_int32


def header_functions() -> list:
    """Names of the functions include/ssd.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(ssd_\w+)\s*\(", text, re.M)))


def library_handle():
    return _lib


def ssd_status_string(status: int) -> str:
    return _lib.ssd_status_string(int(status)).decode()


def ssd_version() -> int:
    return int(_lib.ssd_version())


def make_dims(batch, seqlen, nheads, headdim, dstate, ngroups_b=1, ngroups_c=1,
              io_dtype=SSD_BF16, dt_softplus=True) -> ssd_dims:
    return ssd_dims(int(batch), int(seqlen), int(nheads), int(headdim), int(dstate),
                    int(ngroups_b), int(ngroups_c), int(io_dtype), int(bool(dt_softplus)))


def _io_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SSD_BF16
    if t.dtype == torch.float32:
        return SSD_F32
    raise TypeError("x/B/C must be float32 or bfloat16, got %s" % t.dtype)


def dims_of(x: torch.Tensor, B: torch.Tensor, C: torch.Tensor, dt_softplus=True) -> ssd_dims:
    """Dims from x [b,T,H,P], B [b,T,G_B,N], C [b,T,G_C,N]."""
    b, T, H, P = x.shape
    return make_dims(b, T, H, P, B.shape[3], B.shape[2], C.shape[2], _io_code(x), dt_softplus)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libssd takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libssd takes contiguous tensors")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(status: int, where: str):
    if status != SSD_OK:
        raise SsdError(status, where)


def ssd_fwd_workspace_size(dims: ssd_dims, chunk: int) -> int:
    return int(_lib.ssd_fwd_workspace_size(ctypes.byref(dims), int(chunk)))


def ssd_fwd_num_stages(dims: ssd_dims, chunk: int) -> int:
    return int(_lib.ssd_fwd_num_stages(ctypes.byref(dims), int(chunk)))


def ssd_fwd_stage_name(dims: ssd_dims, chunk: int, i: int) -> Optional[str]:
    r = _lib.ssd_fwd_stage_name(ctypes.byref(dims), int(chunk), int(i))
    return r.decode() if r is not None else None


def _fwd_ptrs(x, dt, A, B, C, D, h0, y, h_final, workspace):
    return [_ptr(t) for t in (x, dt, A, B, C, D, h0)], [_ptr(y), _ptr(h_final), _ptr(workspace)]


def ssd_fwd(x, dt, A, B, C, D, h0, chunk: int, y, h_final, workspace, dt_softplus: bool = True,
            stream=None, dims: Optional[ssd_dims] = None) -> None:
    """Enqueue the chunked SSD forward on `stream` (see ssd.h)."""
    dims = dims or dims_of(x, B, C, dt_softplus)
    ins, outs = _fwd_ptrs(x, dt, A, B, C, D, h0, y, h_final, workspace)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = _lib.ssd_fwd(ctypes.byref(dims), *ins, int(chunk), outs[0], outs[1], outs[2],
                      ws_bytes, _stream(stream))
    _check(st, "ssd_fwd")


def ssd_fwd_profiled(x, dt, A, B, C, D, h0, chunk: int, y, h_final, workspace,
                     events: Sequence[torch.cuda.Event], dt_softplus: bool = True, stream=None,
                     dims: Optional[ssd_dims] = None) -> None:
    """ssd_fwd recording events[i] before stage i and events[-1] after the last."""
    dims = dims or dims_of(x, B, C, dt_softplus)
    n = ssd_fwd_num_stages(dims, chunk)
    if len(events) != n + 1:
        raise ValueError("need %d events" % (n + 1))
    for e in events:          # torch creates the CUDA event lazily
        if e.cuda_event == 0:
            e.record(torch.cuda.current_stream() if stream is None else stream)
    arr = (ctypes.c_void_p * (n + 1))(*[e.cuda_event for e in events])
    ins, outs = _fwd_ptrs(x, dt, A, B, C, D, h0, y, h_final, workspace)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = _lib.ssd_fwd_profiled(ctypes.byref(dims), *ins, int(chunk), outs[0], outs[1], outs[2],
                               ws_bytes, arr, _stream(stream))
    _check(st, "ssd_fwd_profiled")


def ssd_fwd_noalloc(x, dt, A, B, C, D, h0, chunk: int, y, h_final, dt_softplus: bool = True,
                    stream=None, dims: Optional[ssd_dims] = None) -> None:
    """ssd_fwd without a caller workspace: for callers that cannot allocate
    device memory where they run the layer (a fixed memory plan, a framework's
    caching allocator owning the device, or a path that must not pay
    cudaMalloc's implicit synchronisation).  The library's static scratch
    array (SSD_NOALLOC_SCRATCH_BYTES) is used instead; larger shapes raise.
    Calls on one device share that array, so they must not overlap."""
    dims = dims or dims_of(x, B, C, dt_softplus)
    st = _lib.ssd_fwd_noalloc(ctypes.byref(dims), *[_ptr(t) for t in (x, dt, A, B, C, D, h0)],
                              int(chunk), _ptr(y), _ptr(h_final), _stream(stream))
    _check(st, "ssd_fwd_noalloc")


def ssd_multistep(x, dt, A, B, C, D, h_cache, j, y, h_j, h_K, dt_softplus: bool = True,
                  stream=None, dims: Optional[ssd_dims] = None) -> None:
    """Enqueue the K-token verification decode on `stream` (see ssd.h)."""
    dims = dims or dims_of(x, B, C, dt_softplus)
    st = _lib.ssd_multistep(ctypes.byref(dims), *[_ptr(t) for t in (x, dt, A, B, C, D, h_cache, j,
                                                                      y, h_j, h_K)],
                            _stream(stream))
    _check(st, "ssd_multistep")


def ssd_cp_workspace_size(dims: ssd_dims) -> int:
    return int(_lib.ssd_cp_workspace_size(ctypes.byref(dims)))


def ssd_cp_segment_decay(dt, A, decay, workspace, dims: ssd_dims, stream=None) -> None:
    """Enqueue the segment-decay kernels (see ssd.h): decay [b, H] float32."""
    ws_bytes = workspace.numel() * workspace.element_size()
    st = _lib.ssd_cp_segment_decay(ctypes.byref(dims), _ptr(dt), _ptr(A), _ptr(decay),
                                   _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "ssd_cp_segment_decay")


def ssd_cp_correct(nranks: int, rank: int, decays, finals, dt, A, C, y, h_final, workspace,
                   dims: ssd_dims, stream=None) -> None:
    """Enqueue the correction of this rank's segment (see ssd.h)."""
    ws_bytes = workspace.numel() * workspace.element_size()
    st = _lib.ssd_cp_correct(ctypes.byref(dims), int(nranks), int(rank), _ptr(decays),
                             _ptr(finals), _ptr(dt), _ptr(A), _ptr(C), _ptr(y), _ptr(h_final),
                             _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "ssd_cp_correct")


def ssd_selftest_timeout(limit_ns: int, stream=None) -> None:
    """Enqueue the bounded-wait self-test kernel (see ssd.h)."""
    _check(_lib.ssd_selftest_timeout(int(limit_ns), _stream(stream)), "ssd_selftest_timeout")


def ssd_check_device_error(stream=None) -> None:
    """Synchronise and raise if a kernel recorded a device-side error."""
    _check(_lib.ssd_check_device_error(_stream(stream)), "ssd_check_device_error")


# ----------------------------------------------------------------------------- helpers
def workspace_for(dims: ssd_dims, chunk: int, device="cuda") -> torch.Tensor:
    n = ssd_fwd_workspace_size(dims, chunk)
    if n == 0:
        raise SsdError(SSD_ERR_UNSUPPORTED, "ssd_fwd_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def forward(x, dt, A, B, C, D=None, h0=None, chunk: int = 256, dt_softplus: bool = True,
            stream=None):
    """Allocates y, h_final and the workspace with torch and calls ssd_fwd."""
    dims = dims_of(x, B, C, dt_softplus)
    y = torch.empty_like(x)
    b, T, H, P = x.shape
    h_final = torch.empty((b, H, B.shape[3], P), dtype=torch.float32, device=x.device)
    ws = workspace_for(dims, chunk, x.device)
    ssd_fwd(x, dt, A, B, C, D, h0, chunk, y, h_final, ws, dt_softplus, stream, dims)
    return y, h_final


def ssd_fwd_sequential_workspace_size(dims: ssd_dims, chunk: int, window: int) -> int:
    return int(_lib.ssd_fwd_sequential_workspace_size(ctypes.byref(dims), int(chunk), int(window)))


def ssd_fwd_sequential(x, dt, A, B, C, D, h0, chunk: int, window: int, y, h_final, workspace,
                       dt_softplus: bool = True, stream=None,
                       dims: Optional[ssd_dims] = None) -> None:
    """Enqueue the windowed (sequential) prefill on `stream` (see ssd.h)."""
    dims = dims or dims_of(x, B, C, dt_softplus)
    ins, outs = _fwd_ptrs(x, dt, A, B, C, D, h0, y, h_final, workspace)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = _lib.ssd_fwd_sequential(ctypes.byref(dims), *ins, int(chunk), int(window), outs[0],
                                 outs[1], outs[2], ws_bytes, _stream(stream))
    _check(st, "ssd_fwd_sequential")


def forward_sequential(x, dt, A, B, C, D=None, h0=None, chunk: int = 256, window: int = 4096,
                       dt_softplus: bool = True, stream=None):
    """Allocates y, h_final and the (T-independent) workspace; calls ssd_fwd_sequential."""
    dims = dims_of(x, B, C, dt_softplus)
    y = torch.empty_like(x)
    b, T, H, P = x.shape
    h_final = torch.empty((b, H, B.shape[3], P), dtype=torch.float32, device=x.device)
    n = ssd_fwd_sequential_workspace_size(dims, chunk, window)
    if n == 0:
        raise SsdError(SSD_ERR_UNSUPPORTED, "ssd_fwd_sequential_workspace_size")
    ws = torch.empty(n, dtype=torch.uint8, device=x.device)
    ssd_fwd_sequential(x, dt, A, B, C, D, h0, chunk, window, y, h_final, ws, dt_softplus, stream,
                       dims)
    return y, h_final


def ssd_verify(x_prev, dt_prev, B_prev, j_prev, x, dt, A, B, C, D, h_cache, y, h_next,
               dt_softplus: bool = True, stream=None) -> None:
    """Enqueue the fused recompute + decode + cache step on `stream` (see ssd.h).
    The number of previous drafts is x_prev.shape[1]; the new tokens x.shape[1]."""
    dims = dims_of(x, B, C, dt_softplus)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    st = _lib.ssd_verify(ctypes.byref(dims), int(x_prev.shape[1]), p(x_prev), p(dt_prev),
                         p(B_prev), p(j_prev), p(x),
                         p(dt), p(A), p(B), p(C), p(D), p(h_cache), p(y), p(h_next),
                         _stream(stream))
    _check(st, "ssd_verify")


def multistep(x, dt, A, B, C, D, h_cache, j, dt_softplus: bool = True, stream=None):
    """Allocates y, h_j, h_K with torch and calls ssd_multistep."""
    y = torch.empty_like(x)
    h_j = torch.empty_like(h_cache)
    h_K = torch.empty_like(h_cache)
    ssd_multistep(x, dt, A, B, C, D, h_cache, j, y, h_j, h_K, dt_softplus, stream)
    return y, h_j, h_K
