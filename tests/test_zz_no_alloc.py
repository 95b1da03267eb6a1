"""The allocation-free prefill entry point, ssd_fwd_noalloc.

It serves callers that cannot call cudaMalloc where they run the layer: code
under a fixed device-memory plan, code inside a framework whose caching
allocator owns the device memory, and latency-critical paths that cannot take
cudaMalloc's implicit synchronisation.  Instead of a caller workspace it uses
the library's static device scratch array.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.  It must pass alone in a fresh
process and after the rest of the suite.
"""
import ctypes

import pytest
import torch

from state_space_model_09_b300 import ssd as S
from state_space_model_09_b300 import synth

pytestmark = pytest.mark.gpu

NOALLOC_SCRATCH_BYTES = 64 << 20  # SSD_NOALLOC_SCRATCH_BYTES in include/ssd.h
TOL = {synth.F32: 1e-4, synth.BF16: 1e-2}


def _device_inputs(shape, seed):
    inp = synth.make_fwd_inputs(shape, seed)
    io_t = torch.bfloat16 if shape.io == synth.BF16 else torch.float32
    d = {}
    for k, v in inp.items():
        if v is None:
            d[k] = None
        else:
            t = torch.from_numpy(v).cuda()
            d[k] = t.to(io_t) if k in ("x", "B", "C") else t
    return d


def _call_noalloc(d, chunk, y, h_final):
    """Calls ssd_fwd_noalloc straight through the C ABI (ctypes)."""
    lib = S.library_handle()
    dims = S.dims_of(d["x"], d["B"], d["C"])
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.ssd_fwd_noalloc(ctypes.byref(dims), ptr(d["x"]), ptr(d["dt"]), ptr(d["A"]),
                               ptr(d["B"]), ptr(d["C"]), ptr(d["D"]), ptr(d["h0"]), int(chunk),
                               ptr(y), ptr(h_final), stream)


def _rel(a, b):
    a, b = a.double(), b.double()
    return float((a - b).abs().max() / b.abs().max())


@pytest.mark.parametrize("shape,seed", [
    # tensor-core path (bf16, Q = 256, ragged last chunk, random h0)
    (synth.FwdShape(2, 600, 4, 64, 128, 1, 1, 256, synth.BF16, "all"), 91),
    # float32 path (the tiny workload's kernels)
    (synth.FwdShape(1, 256, 4, 64, 64, 1, 1, 64, synth.F32, "zero"), 92),
])
def test_noalloc_matches_workspace_entry_point(shape, seed):
    d = _device_inputs(shape, seed)
    dims = S.dims_of(d["x"], d["B"], d["C"])
    assert 0 < S.ssd_fwd_workspace_size(dims, shape.chunk) <= NOALLOC_SCRATCH_BYTES

    # the existing entry point, with a caller-owned workspace
    y_ref, h_ref = S.forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"],
                             chunk=shape.chunk)
    torch.cuda.synchronize()

    b, T, H, P = d["x"].shape
    N = d["B"].shape[3]
    # two calls in a row: the second reuses the first call's scratch contents
    for _ in range(2):
        y = torch.full_like(d["x"], float("nan"))
        hf = torch.full((b, H, N, P), float("nan"), device="cuda")
        assert _call_noalloc(d, shape.chunk, y, hf) == S.SSD_OK
        S.ssd_check_device_error()
        assert torch.isfinite(y.float()).all() and torch.isfinite(hf).all()
        assert _rel(y, y_ref) <= TOL[shape.io]
        assert _rel(hf, h_ref) <= TOL[shape.io]


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # a Mamba-2 2.7B layer needs ~257 MB of scratch, above the static array
    shape = synth.FwdShape(8, 2048, 80, 64, 128, 1, 1, 256, synth.BF16, "zero")
    dims = S.make_dims(8, 2048, 80, 64, 128)
    assert S.ssd_fwd_workspace_size(dims, 256) > NOALLOC_SCRATCH_BYTES
    x = torch.zeros((8, 2048, 80, 64), dtype=torch.bfloat16, device="cuda")
    Bm = torch.zeros((8, 2048, 1, 128), dtype=torch.bfloat16, device="cuda")
    Cm = torch.zeros_like(Bm)
    dt = torch.zeros((8, 2048, 80), device="cuda")
    A = torch.zeros(80, device="cuda")
    d = dict(x=x, dt=dt, A=A, B=Bm, C=Cm, D=None, h0=None)
    y = torch.empty_like(x)
    assert _call_noalloc(d, shape.chunk, y, None) == S.SSD_ERR_UNSUPPORTED
