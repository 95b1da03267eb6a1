"""fp64 CPU oracle for the SSD layer and the multi-step decode.

TEST INFRASTRUCTURE: imported only by tests/, the smoke check and the
benchmark's CPU-baseline / reference leg.  The product path (the CUDA library
and its binding) never imports it.

The C source is ssd_oracle.c; this module only marshals numpy arrays.  Results
are returned in "pair-compact" form: the leading axis enumerates the requested
(b, h) pairs (q -> b*H + h), e.g. y[q, t, p] and h[q, n, p].
"""
from __future__ import annotations

import ctypes
import threading
from typing import Optional, Sequence

import numpy as np

from .build import build_oracle

_lib = None
_lock = threading.Lock()

_f = ctypes.POINTER(ctypes.c_float)
_d = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build_oracle())
            common = [_i64] * 7 + [ctypes.c_void_p] * 7
            lib.oracle_ssd_seq.argtypes = common + [ctypes.c_int, ctypes.c_void_p, _i64,
                                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.oracle_ssd_chunked.argtypes = common + [ctypes.c_int, _i64, ctypes.c_void_p, _i64,
                                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.oracle_ssd_multistep.argtypes = common + [ctypes.c_void_p, ctypes.c_int,
                                                          ctypes.c_void_p, _i64, ctypes.c_void_p,
                                                          ctypes.c_void_p, ctypes.c_void_p,
                                                          ctypes.c_int]
            for fn in (lib.oracle_ssd_seq, lib.oracle_ssd_chunked, lib.oracle_ssd_multistep):
                fn.restype = ctypes.c_int
            lib.oracle_default_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    return _load().oracle_default_threads()


def _f32(a):
    if a is None:
        return None, None
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _pairs(pairs, batch, H):
    if pairs is None:
        return None, None, batch * H
    p = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64))
    assert p.ndim == 1 and (p >= 0).all() and (p < batch * H).all()
    return p, p.ctypes.data_as(ctypes.c_void_p), len(p)


def _common(x, dt, A, B, C, D, h0):
    keep = [_f32(v) for v in (x, dt, A, B, C, D, h0)]
    return keep, [k[1] for k in keep]


def ssd_seq(x, dt, A, B, C, D=None, h0=None, dt_softplus: bool = True,
            pairs: Optional[Sequence[int]] = None, nthreads: int = 0):
    """Sequential fp64 recurrence.  x [b,T,H,P], dt [b,T,H], B [b,T,G_B,N],
    C [b,T,G_C,N], A/D [H], h0 [b,H,N,P] or None.  Returns (y[q,T,P], h[q,N,P])."""
    b, T, H, P = x.shape
    GB, N = B.shape[2], B.shape[3]
    GC = C.shape[2]
    keep, ptrs = _common(x, dt, A, B, C, D, h0)
    pk, pp, npairs = _pairs(pairs, b, H)
    y = np.empty((npairs, T, P), dtype=np.float64)
    hf = np.empty((npairs, N, P), dtype=np.float64)
    rc = _load().oracle_ssd_seq(b, T, H, P, N, GB, GC, *ptrs, int(dt_softplus), pp, npairs,
                                y.ctypes.data_as(ctypes.c_void_p),
                                hf.ctypes.data_as(ctypes.c_void_p), nthreads)
    if rc:
        raise ValueError("oracle_ssd_seq rejected its arguments (rc=%d)" % rc)
    del keep, pk
    return y, hf


def ssd_chunked(x, dt, A, B, C, D=None, h0=None, chunk: int = 64, dt_softplus: bool = True,
                pairs: Optional[Sequence[int]] = None, nthreads: int = 0):
    """Chunked block decomposition in fp64 (same layouts and outputs as ssd_seq)."""
    b, T, H, P = x.shape
    GB, N = B.shape[2], B.shape[3]
    GC = C.shape[2]
    keep, ptrs = _common(x, dt, A, B, C, D, h0)
    pk, pp, npairs = _pairs(pairs, b, H)
    y = np.empty((npairs, T, P), dtype=np.float64)
    hf = np.empty((npairs, N, P), dtype=np.float64)
    rc = _load().oracle_ssd_chunked(b, T, H, P, N, GB, GC, *ptrs, int(dt_softplus), int(chunk),
                                    pp, npairs, y.ctypes.data_as(ctypes.c_void_p),
                                    hf.ctypes.data_as(ctypes.c_void_p), nthreads)
    if rc:
        raise ValueError("oracle_ssd_chunked rejected its arguments (rc=%d)" % rc)
    del keep, pk
    return y, hf


def ssd_multistep(x, dt, A, B, C, D, h_cache, j, dt_softplus: bool = True,
                  pairs: Optional[Sequence[int]] = None, nthreads: int = 0):
    """K steps from h_cache.  x [b,K,H,P], dt [b,K,H], B/C [b,K,G,N], h_cache
    [b,H,N,P], j [b] in 0..K.  Returns (y[q,K,P], h_j[q,N,P], h_K[q,N,P])."""
    b, K, H, P = x.shape
    GB, N = B.shape[2], B.shape[3]
    GC = C.shape[2]
    keep, ptrs = _common(x, dt, A, B, C, D, h_cache)
    jj = np.ascontiguousarray(np.asarray(j, dtype=np.int32))
    pk, pp, npairs = _pairs(pairs, b, H)
    y = np.empty((npairs, K, P), dtype=np.float64)
    hj = np.empty((npairs, N, P), dtype=np.float64)
    hK = np.empty((npairs, N, P), dtype=np.float64)
    rc = _load().oracle_ssd_multistep(b, K, H, P, N, GB, GC, *ptrs,
                                      jj.ctypes.data_as(ctypes.c_void_p), int(dt_softplus), pp,
                                      npairs, y.ctypes.data_as(ctypes.c_void_p),
                                      hj.ctypes.data_as(ctypes.c_void_p),
                                      hK.ctypes.data_as(ctypes.c_void_p), nthreads)
    if rc:
        raise ValueError("oracle_ssd_multistep rejected its arguments (rc=%d)" % rc)
    del keep, pk
    return y, hj, hK


def to_full(y_pairs: np.ndarray, batch: int, H: int) -> np.ndarray:
    """Pair-compact y[q,T,P] (all pairs, in order) -> y[b,T,H,P]."""
    q, T, P = y_pairs.shape
    assert q == batch * H
    return y_pairs.reshape(batch, H, T, P).transpose(0, 2, 1, 3).copy()


def states_full(h_pairs: np.ndarray, batch: int, H: int) -> np.ndarray:
    """Pair-compact h[q,N,P] (all pairs) -> h[b,H,N,P]."""
    q, N, P = h_pairs.shape
    return h_pairs.reshape(batch, H, N, P)
