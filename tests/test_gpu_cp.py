"""Context parallelism on one GPU: a sequence cut into segments, each run
through ssd_fwd from a zero state (the first from h0), the segment decays
and final states stacked in rank order, then every segment corrected with
ssd_cp_correct.  The concatenated outputs equal the oracle's whole-sequence
outputs and every segment's corrected final state equals the oracle's state
at that segment's end (the last one: the sequence's final state)."""
import numpy as np
import pytest
import torch

import oracle
from state_space_model_09_b300 import ssd as S
from state_space_model_09_b300 import synth

pytestmark = pytest.mark.gpu

F = synth.FwdShape
TOL = {synth.F32: 1e-4, synth.BF16: 1e-2}


def _dev(a, io=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    if io == synth.BF16:
        t = t.to(torch.bfloat16)
    return t


def run_segments(shape, inp, cuts, dt_softplus=True):
    """Returns (y [b, T, H, P] float32 numpy, [h_final of every segment])."""
    bounds = [0] + list(cuts) + [shape.seqlen]
    segs = []
    for r in range(len(bounds) - 1):
        sl = slice(bounds[r], bounds[r + 1])
        d = dict(x=_dev(inp["x"][:, sl], shape.io), dt=_dev(inp["dt"][:, sl]),
                 B=_dev(inp["B"][:, sl], shape.io), C=_dev(inp["C"][:, sl], shape.io))
        segs.append(d)
    A = _dev(inp["A"])
    D = None if inp["D"] is None else _dev(inp["D"])
    h0 = None if inp["h0"] is None else _dev(inp["h0"])
    R = len(segs)
    ys, decays, finals, dims_l, wss = [], [], [], [], []
    for r, d in enumerate(segs):
        y, hf = S.forward(d["x"], d["dt"], A, d["B"], d["C"], D, h0 if r == 0 else None,
                          chunk=shape.chunk, dt_softplus=dt_softplus)
        dims = S.dims_of(d["x"], d["B"], d["C"], dt_softplus)
        ws = torch.empty(S.ssd_cp_workspace_size(dims), dtype=torch.uint8, device="cuda")
        ws.fill_(0xFF)  # NaN-poisoned scratch
        dec = torch.empty((shape.batch, shape.nheads), device="cuda")
        S.ssd_cp_segment_decay(d["dt"], A, dec, ws, dims)
        ys.append(y)
        decays.append(dec)
        finals.append(hf)
        dims_l.append(dims)
        wss.append(ws)
    decays = torch.stack(decays).contiguous()
    finals = torch.stack(finals).contiguous()
    outs = []
    for r, d in enumerate(segs):
        hf = torch.full_like(finals[0], float("nan"))
        S.ssd_cp_correct(R, r, decays, finals, d["dt"], A, d["C"], ys[r], hf, wss[r], dims_l[r])
        outs.append(hf)
    torch.cuda.synchronize()
    S.ssd_check_device_error()
    y = torch.cat([t.float() for t in ys], dim=1).cpu().numpy()
    return y, [h.cpu().numpy() for h in outs], bounds


def check(shape, seed, cuts, pairs=None, dt_softplus=True):
    inp = synth.make_fwd_inputs(shape, seed)
    if not dt_softplus:
        inp["dt"] = np.abs(inp["dt"]) * np.float32(0.05)
    y, finals, bounds = run_segments(shape, inp, cuts, dt_softplus)
    H = shape.nheads
    pairs = pairs or list(range(shape.batch * H))
    yr, hr = oracle.ssd_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"],
                            dt_softplus=dt_softplus, pairs=pairs)
    tol = TOL[shape.io]
    ys = np.stack([y[p // H, :, p % H, :] for p in pairs]).astype(np.float64)
    assert np.abs(ys - yr).max() / np.abs(yr).max() <= tol
    # each segment's corrected final state = the state after its last token
    for r in range(len(bounds) - 1):
        end = bounds[r + 1]
        if end == shape.seqlen:
            ref = hr
        else:
            cut = {k: (v[:, :end] if k in ("x", "dt", "B", "C") else v) for k, v in inp.items()}
            _, ref = oracle.ssd_seq(cut["x"], cut["dt"], cut["A"], cut["B"], cut["C"], cut["D"],
                                    cut["h0"], dt_softplus=dt_softplus, pairs=pairs)
        got = np.stack([finals[r][p // H, p % H] for p in pairs]).astype(np.float64)
        assert np.abs(got - ref).max() / np.abs(ref).max() <= tol, r


@pytest.mark.parametrize("shape,seed,cuts", [
    # tensor-core correction, 64-wide heads, one group, uneven segments
    (F(2, 1000, 4, 64, 128, 1, 1, 256, synth.BF16, "all"), 91, (300, 750)),
    # 128-wide heads, grouped B and C (C group per pair of heads), chunk 128
    (F(2, 600, 8, 128, 128, 2, 4, 128, synth.BF16, "all"), 92, (257,)),
    # float32 path (CUDA-core correction), four segments, one of a single token
    (F(1, 300, 3, 32, 32, 1, 1, 64, synth.F32, "all"), 93, (64, 65, 200)),
    # bf16 outside the tensor-core envelope (N = 64)
    (F(2, 200, 4, 64, 64, 1, 2, 64, synth.BF16, "zero"), 94, (100,)),
    # tensor-core correction on segments of exactly one tile, one token, one
    # token short of a tile, and one tile and a bit
    (F(1, 400, 4, 64, 128, 1, 1, 256, synth.BF16, "all"), 99, (128, 129, 256)),
])
def test_segments_equal_whole_sequence(shape, seed, cuts):
    check(shape, seed, cuts)


def test_segments_without_softplus():
    check(F(1, 500, 4, 64, 128, 1, 1, 256, synth.BF16, "all"), 95, (256,), dt_softplus=False)


def test_long_16k_in_two_segments_sampled():
    """The 16K-token workload split at 8192 tokens: sampled (b, h) pairs."""
    shape = synth.WORKLOADS["long_16k"]
    check(shape, synth.WORKLOAD_SEEDS["long_16k"], (8192,), pairs=[0, 7, 33, 40, 79])


def test_long_16k_in_three_uneven_segments_sampled():
    """Segments of 5000, 6000 and 5384 tokens: the tensor-core correction runs
    several heads per CTA (its two-deep head pipeline) over ragged last
    tiles."""
    shape = synth.WORKLOADS["long_16k"]
    check(shape, synth.WORKLOAD_SEEDS["long_16k"], (5000, 11000), pairs=[1, 6, 38, 64, 79])


@pytest.mark.parametrize("shape,seed,cuts,pairs", [
    # the 2.7B layer's heads, four batch rows: the correction's units run two
    # heads each and span batch rows, over ragged last tiles
    (F(4, 4096, 80, 64, 128, 1, 1, 256, synth.BF16, "half"), 97, (1500, 2900),
     [3, 81, 170, 259, 319]),
    # 128-wide heads (P = 128) over a long sequence: two heads per unit
    (F(1, 8192, 64, 128, 128, 1, 1, 128, synth.BF16, "all"), 98, (3000,), [0, 17, 40, 63]),
])
def test_large_segments_sampled(shape, seed, cuts, pairs):
    check(shape, seed, cuts, pairs=pairs)


def test_rank0_leaves_y_and_copies_its_final_state():
    shape = F(1, 300, 2, 64, 128, 1, 1, 256, synth.BF16, "all")
    inp = synth.make_fwd_inputs(shape, 96)
    d = {k: (None if v is None else _dev(v, shape.io if k in ("x", "B", "C") else None))
         for k, v in inp.items()}
    y, hf = S.forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"], chunk=256)
    dims = S.dims_of(d["x"], d["B"], d["C"])
    ws = torch.empty(S.ssd_cp_workspace_size(dims), dtype=torch.uint8, device="cuda")
    dec = torch.empty((1, 2), device="cuda")
    S.ssd_cp_segment_decay(d["dt"], d["A"], dec, ws, dims)
    y0 = y.clone()
    out = torch.empty_like(hf)
    S.ssd_cp_correct(2, 0, torch.stack([dec, dec]), torch.stack([hf, hf]), d["dt"], d["A"],
                     d["C"], y, out, ws, dims)
    torch.cuda.synchronize()
    assert torch.equal(y, y0) and torch.equal(out, hf)
    # the segment decay is the product of the tokens' exp(softplus(dt) A)
    dtd = inp["dt"].astype(np.float64)
    sp = np.where(dtd > 20, dtd, np.log1p(np.exp(np.minimum(dtd, 20))))
    ref = np.exp((sp * inp["A"].astype(np.float64)[None, None, :]).sum(axis=1))
    assert np.allclose(dec.cpu().numpy(), ref, rtol=1e-4, atol=1e-30)
