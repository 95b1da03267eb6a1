"""Sequential (chunked-prompt) prefill: ssd_fwd_sequential processes a prompt
in windows chained through the state, in device memory that does not grow
with the prompt length.  It must equal one ssd_fwd over the whole sequence
(up to rounding) and the oracle, for contiguous windows (batch 1) and for
windows gathered from batched tensors (batch > 1)."""
import numpy as np
import pytest
import torch

import oracle
from state_space_model_09_b300 import ssd as S
from state_space_model_09_b300 import synth

pytestmark = pytest.mark.gpu

F = synth.FwdShape
TOL = {synth.F32: 1e-4, synth.BF16: 1e-2}


def _dev(inp, io):
    dt_io = torch.bfloat16 if io == synth.BF16 else torch.float32
    return {k: (None if v is None else
                torch.from_numpy(v).to(dt_io).cuda() if k in ("x", "B", "C") else
                torch.from_numpy(v).cuda())
            for k, v in inp.items()}


def _rel(a, b):
    a, b = a.double(), b.double()
    return float((a - b).abs().max() / b.abs().max())


@pytest.mark.parametrize("shape,window,seed", [
    (F(1, 1000, 4, 64, 128, 1, 1, 256, synth.BF16, "all"), 256, 81),   # contiguous windows
    (F(2, 900, 4, 64, 128, 1, 2, 128, synth.BF16, "half"), 300, 82),   # staged, off the chunk grid
    (F(3, 700, 4, 32, 32, 1, 1, 64, synth.F32, "all"), 192, 83),       # float32 path, staged
    (F(1, 130, 2, 64, 64, 1, 1, 64, synth.F32, "zero"), 1000, 84),     # window longer than T
    (F(1, 1000, 3, 64, 128, 1, 1, 256, synth.BF16, "all"), 250, 86),   # dt windows staged (H = 3)
])
def test_sequential_equals_whole_and_oracle(shape, window, seed):
    inp = synth.make_fwd_inputs(shape, seed)
    d = _dev(inp, shape.io)
    y_whole, h_whole = S.forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"],
                                 chunk=shape.chunk)
    y_seq, h_seq = S.forward_sequential(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"],
                                        chunk=shape.chunk, window=window)
    torch.cuda.synchronize()
    S.ssd_check_device_error()
    tol = TOL[shape.io]
    assert _rel(y_seq.float(), y_whole.float()) <= tol
    assert _rel(h_seq, h_whole) <= tol
    # against the oracle on every (b, h) pair
    H = shape.nheads
    pairs = list(range(shape.batch * H))
    y_ref, h_ref = oracle.ssd_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                                  inp["h0"], pairs=pairs)
    yy = y_seq.float().cpu().numpy().astype(np.float64)
    ys = np.stack([yy[p // H, :, p % H, :] for p in pairs])
    hh = h_seq.cpu().numpy().astype(np.float64)
    hs = np.stack([hh[p // H, p % H] for p in pairs])
    assert np.abs(ys - y_ref).max() / np.abs(y_ref).max() <= tol
    assert np.abs(hs - h_ref).max() / np.abs(h_ref).max() <= tol


def test_sequential_without_h0_and_h_final_graph_replay():
    """NULL h0 / h_final, and the whole windowed call captured in a CUDA graph
    replays to the eager result bit for bit."""
    shape = F(2, 600, 4, 64, 128, 1, 1, 256, synth.BF16, "zero")
    d = _dev(synth.make_fwd_inputs(shape, 85), shape.io)
    dims = S.dims_of(d["x"], d["B"], d["C"])
    window = 256
    ws = torch.empty(S.ssd_fwd_sequential_workspace_size(dims, 256, window), dtype=torch.uint8,
                     device="cuda")
    y_ref = torch.empty_like(d["x"])
    S.ssd_fwd_sequential(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], None, 256, window, y_ref,
                         None, ws)
    torch.cuda.synchronize()
    y = torch.empty_like(d["x"])
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        S.ssd_fwd_sequential(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], None, 256, window,
                             y, None, ws, stream=stream)
    for _ in range(2):
        y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref)
