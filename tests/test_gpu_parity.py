"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Tolerance (the layer's stated bar): max|y - y_ref| / max|y_ref| <= 1e-2 with
bf16 inputs and float32 state, <= 1e-4 with float32 inputs; the same bound on
every returned state.  Small shapes are compared element by element over the
whole output; the full-size workloads are compared on sampled (b, h) pairs,
which the oracle computes independently of the others.
"""
import numpy as np
import pytest
import torch

import oracle
from state_space_model_09_b300 import ssd as S
from state_space_model_09_b300 import synth

pytestmark = pytest.mark.gpu

TOL = {synth.F32: 1e-4, synth.BF16: 1e-2}


def rel_err(got, ref):
    return float(np.abs(got - ref).max() / np.abs(ref).max())


def to_dev(inp, io):
    dt_io = torch.bfloat16 if io == synth.BF16 else torch.float32
    out = {}
    for k, v in inp.items():
        if v is None:
            out[k] = None
        elif k in ("x", "B", "C"):
            out[k] = torch.from_numpy(v).to(dt_io).cuda()
        elif k == "j":
            out[k] = torch.from_numpy(v).cuda()
        else:
            out[k] = torch.from_numpy(v).cuda()
    return out


def run_fwd(d, chunk, dt_softplus=True, with_final=True):
    y = torch.full_like(d["x"], float("nan"))
    b, T, H, P = d["x"].shape
    N = d["B"].shape[3]
    hf = torch.full((b, H, N, P), float("nan"), device="cuda") if with_final else None
    dims = S.dims_of(d["x"], d["B"], d["C"], dt_softplus)
    ws = S.workspace_for(dims, chunk)
    ws.fill_(0xFF)  # NaN-poison the scratch
    S.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"], chunk, y, hf, ws,
              dt_softplus)
    S.ssd_check_device_error()
    return y, hf


def y_pairs(y, pairs, H):
    """y [b,T,H,P] (torch) -> [len(pairs), T, P] float64 numpy."""
    yy = y.float().cpu().numpy().astype(np.float64)
    return np.stack([yy[p // H, :, p % H, :] for p in pairs])


def h_pairs(h, pairs, H):
    hh = h.cpu().numpy().astype(np.float64)
    return np.stack([hh[p // H, p % H] for p in pairs])


def check_fwd(shape, seed, pairs=None, dt_softplus=True, D_none=False):
    inp = synth.make_fwd_inputs(shape, seed)
    if D_none:
        inp["D"] = None
    if not dt_softplus:
        inp["dt"] = np.abs(inp["dt"]) * np.float32(0.05)
    d = to_dev(inp, shape.io)
    y, hf = run_fwd(d, shape.chunk, dt_softplus)
    H = shape.nheads
    if pairs is None:
        pairs = list(range(shape.batch * H))
    y_ref, h_ref = oracle.ssd_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                                  inp["h0"], dt_softplus=dt_softplus, pairs=pairs)
    ey = rel_err(y_pairs(y, pairs, H), y_ref)
    eh = rel_err(h_pairs(hf, pairs, H), h_ref)
    tol = TOL[shape.io]
    assert np.isfinite(ey) and np.isfinite(eh)
    assert ey <= tol, "y rel err %.3g > %.1g" % (ey, tol)
    assert eh <= tol, "h_final rel err %.3g > %.1g" % (eh, tol)
    return ey, eh


F = synth.FwdShape

SMALL = {
    # float32 I/O (CUDA-core float32 kernels)
    "tiny_f32": (synth.WORKLOADS["tiny_f32"], 1000),
    "f32_ragged_groups": (F(2, 200, 4, 48, 32, 2, 4, 64, synth.F32, "all"), 11),
    "f32_T1": (F(1, 1, 2, 16, 16, 1, 1, 64, synth.F32, "all"), 12),
    "f32_q128_short": (F(1, 100, 2, 32, 64, 1, 2, 128, synth.F32, "zero"), 13),
    # bf16 I/O on the tensor-core kernels
    "tc_q256_p64": (F(2, 600, 4, 64, 128, 1, 1, 256, synth.BF16, "all"), 21),
    "tc_q256_exact": (F(1, 512, 3, 64, 128, 1, 1, 256, synth.BF16, "zero"), 22),
    "tc_q128_p128_groups": (F(2, 300, 8, 128, 128, 2, 8, 128, synth.BF16, "half"), 23),
    "tc_q128_p64": (F(1, 384, 4, 64, 128, 1, 4, 128, synth.BF16, "all"), 24),
    "tc_T1": (F(1, 1, 2, 64, 128, 1, 1, 256, synth.BF16, "all"), 25),
    "tc_T_short": (F(2, 77, 2, 64, 128, 1, 2, 256, synth.BF16, "all"), 26),
    # few (batch, head) pairs and many chunks: the state pass runs in sequence
    # segments joined by state_fixup (ragged last chunk, random h0)
    "tc_segments_q128": (F(1, 2000, 2, 64, 128, 1, 1, 128, synth.BF16, "all"), 27),
    "tc_segments_q256": (F(1, 3000, 3, 64, 128, 1, 1, 256, synth.BF16, "all"), 28),
    # bf16 I/O outside the tensor-core envelope (float32 CUDA-core kernels)
    "bf16_q64_n64": (F(2, 160, 4, 64, 64, 1, 1, 64, synth.BF16, "all"), 31),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_fwd_small(name):
    shape, seed = SMALL[name]
    check_fwd(shape, seed)


# small 256-token, single-group cases, also forced through the head-pair form
# (the call picks it only when each CTA gets enough head pairs)
PAIR_FORM = ["tc_q256_p64", "tc_q256_exact", "tc_T1", "tc_segments_q256"]


@pytest.mark.parametrize("name", PAIR_FORM)
def test_fwd_small_pair_form(name, monkeypatch):
    monkeypatch.setenv("SSD_CHUNK_SCAN", "pair")
    shape, seed = SMALL[name]
    d = S.make_dims(shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate,
                    shape.ngroups_b, shape.ngroups_c)
    assert "chunk_scan_hb" in [S.ssd_fwd_stage_name(d, shape.chunk, i)
                               for i in range(S.ssd_fwd_num_stages(d, shape.chunk))]
    check_fwd(shape, seed)


def chunk_log2_decays(inp, Q):
    """Total log2 decay of every (batch, chunk, head): sum over the chunk's
    tokens of softplus(dt) A log2(e) (a property of the inputs, to check that
    a test reaches the decay ranges it is meant to)."""
    dt = inp["dt"].astype(np.float64)
    sp = np.where(dt > 20, dt, np.log1p(np.exp(np.minimum(dt, 20))))
    a = sp * inp["A"].astype(np.float64)[None, None, :] / np.log(2.0)
    b, T, H = a.shape
    nc = -(-T // Q)
    a = np.pad(a, ((0, 0), (0, nc * Q - T), (0, 0)))
    return a.reshape(b, nc, Q, H).sum(axis=2)


def set_form(monkeypatch, form):
    """fused: the one-pass kernel (forced; the default when the items fill a
    wave of the SMs); pair / head: the two-pass head-pair kernels with the
    chunk-scan form forced."""
    if form == "fused":
        monkeypatch.delenv("SSD_CHUNK_SCAN", raising=False)
        monkeypatch.setenv("SSD_FUSED", "1")
    else:
        monkeypatch.setenv("SSD_CHUNK_SCAN", form)


@pytest.mark.parametrize("form", ["fused", "pair", "head"])
@pytest.mark.parametrize("a_scale,window", [
    ((30.0, 1.0, 30.0, 1.0, 1.0), None),       # heads 0 and 2 decay past the scaled form's range
    ((30.0, 30.0, 30.0, 30.0, 30.0), None),    # every head does
    ((0.01, 0.01, 0.01, 0.01, 0.01), None),    # none does
    ((2.5, 2.0, 1.5, 3.0, 1.0), (-192, -96)),  # decays needing a shifted reference
])
def test_fwd_q256_long_decay_heads(a_scale, window, form, monkeypatch):
    """256-token chunks of one group: chunks whose total decay is below 2^-96
    take the scaled form with a shifted reference (factors 2^(r - a_j) and
    2^(a_i - r), the chunk state stored times 2^r); below 2^-192 they are
    flagged by the chunk-state kernel and computed one by one in the head-pair
    launch; either way, and with the head-by-head kernel throughout, every
    head's y and state match the oracle (odd head count, so one pair has a
    single head; ragged last chunk; random h0).  The one-pass kernel applies
    the same range test to each 128-token half of a chunk and leaves the
    chunks that fail it to the per-head body."""
    set_form(monkeypatch, form)
    shape = F(2, 700, 5, 64, 128, 1, 1, 256, synth.BF16, "all")
    inp = synth.make_fwd_inputs(shape, 41)
    inp["A"] = (inp["A"] * np.asarray(a_scale, dtype=np.float32)).astype(np.float32)
    if window:
        al = chunk_log2_decays(inp, shape.chunk)
        assert ((al > window[0]) & (al < window[1])).any(), al
    d = to_dev(inp, shape.io)
    y, hf = run_fwd(d, shape.chunk)
    pairs = list(range(shape.batch * shape.nheads))
    y_ref, h_ref = oracle.ssd_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                                  inp["h0"], pairs=pairs)
    ey = rel_err(y_pairs(y, pairs, shape.nheads), y_ref)
    eh = rel_err(h_pairs(hf, pairs, shape.nheads), h_ref)
    assert np.isfinite(ey) and ey <= TOL[synth.BF16], ey
    assert np.isfinite(eh) and eh <= TOL[synth.BF16], eh


@pytest.mark.parametrize("form", ["pair", "head"])
def test_fwd_q256_last_wave_split_into_segments(form, monkeypatch):
    """4 x 40 head pairs on 148 SMs: the chunk-state kernel runs 148 items
    whole and splits the last 12 (batch 3, heads 56-79) into sequence
    segments joined by the fix-up; heads on both sides of the boundary match
    the oracle (random h0 everywhere, so segment 0 of a split item starts
    from it), with either chunk-scan form after it."""
    monkeypatch.setenv("SSD_CHUNK_SCAN", form)
    shape = F(4, 1024, 80, 64, 128, 1, 1, 256, synth.BF16, "all")
    d = S.make_dims(shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate)
    names = [S.ssd_fwd_stage_name(d, 256, i) for i in range(S.ssd_fwd_num_stages(d, 256))]
    scan = "chunk_scan_hb" if form == "pair" else "chunk_scan_hl"
    assert names == ["dt_decay", "chunk_state_hb", "state_fixup", scan]
    H = shape.nheads
    pairs = [0, 1, 2 * H + 79, 3 * H + 54, 3 * H + 55, 3 * H + 56, 3 * H + 57, 3 * H + 70,
             3 * H + 79]
    check_fwd(shape, 29, pairs=pairs)


def test_fwd_fused_last_wave_split_into_segments(monkeypatch):
    """One-pass kernel, 4 x 40 head pairs on 148 SMs: 148 items run whole, the
    last 12 in four one-chunk segments whose entering states come from the
    prepass; heads on both sides of the boundary match the oracle."""
    set_form(monkeypatch, "fused")
    shape = F(4, 1024, 80, 64, 128, 1, 1, 256, synth.BF16, "all")
    d = S.make_dims(shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate)
    names = [S.ssd_fwd_stage_name(d, 256, i) for i in range(S.ssd_fwd_num_stages(d, 256))]
    assert names == ["chunk_fused_prepass", "chunk_fused_hb", "chunk_scan_flagged"]
    H = shape.nheads
    pairs = [0, 1, 2 * H + 79, 3 * H + 54, 3 * H + 55, 3 * H + 56, 3 * H + 57, 3 * H + 70,
             3 * H + 79]
    check_fwd(shape, 29, pairs=pairs)


def test_fwd_fused_16_byte_aligned_state_buffers(monkeypatch):
    """The one-pass kernel moves a state row in 32-byte accesses where the row
    is 32-byte aligned and in 16-byte ones otherwise: h0, h_final and a
    workspace (holding the segments' states) that are only 16-byte aligned
    give the same bits as 256-byte aligned ones."""
    set_form(monkeypatch, "fused")
    shape = F(4, 1024, 80, 64, 128, 1, 1, 256, synth.BF16, "all")  # a split last wave
    d = to_dev(synth.make_fwd_inputs(shape, 45), shape.io)
    y1, h1 = run_fwd(d, 256)
    b, T, H, P = d["x"].shape
    N = d["B"].shape[3]
    dims = S.dims_of(d["x"], d["B"], d["C"])
    nws = S.ssd_fwd_workspace_size(dims, 256)
    ws_big = torch.full((nws + 64,), 0xFF, dtype=torch.uint8, device="cuda")
    ws = ws_big[16:16 + nws]
    h0_big = torch.empty(d["h0"].numel() + 4, device="cuda")
    h0 = h0_big[4:].view_as(d["h0"])
    h0.copy_(d["h0"])
    hf_big = torch.full((h1.numel() + 4,), float("nan"), device="cuda")
    hf = hf_big[4:].view_as(h1)
    assert h0.data_ptr() % 32 == 16 and hf.data_ptr() % 32 == 16 and ws.data_ptr() % 32 == 16
    y2 = torch.full_like(y1, float("nan"))
    S.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], h0, 256, y2, hf, ws)
    S.ssd_check_device_error()
    assert torch.equal(y1, y2)
    assert torch.equal(h1, hf)


@pytest.mark.parametrize("shape,seed", [
    (F(1, 3000, 3, 64, 128, 1, 1, 256, synth.BF16, "all"), 30),   # 12 one-chunk segments
    (F(3, 1000, 37, 64, 128, 1, 1, 256, synth.BF16, "half"), 31),  # odd H, 2 segments
    (F(2, 129, 2, 64, 128, 1, 1, 256, synth.BF16, "all"), 32),    # one token in the second stage
])
def test_fwd_fused_segments_and_ragged(shape, seed, monkeypatch):
    set_form(monkeypatch, "fused")
    check_fwd(shape, seed)


def check_fwd_scaled_A(shape, seed, a_scale):
    """check_fwd with A multiplied by a_scale (longer decays)."""
    inp = synth.make_fwd_inputs(shape, seed)
    inp["A"] = (inp["A"] * np.float32(a_scale)).astype(np.float32)
    d = to_dev(inp, shape.io)
    y, hf = run_fwd(d, shape.chunk)
    pairs = list(range(shape.batch * shape.nheads))
    y_ref, h_ref = oracle.ssd_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                                  inp["h0"], pairs=pairs)
    ey = rel_err(y_pairs(y, pairs, shape.nheads), y_ref)
    eh = rel_err(h_pairs(hf, pairs, shape.nheads), h_ref)
    assert np.isfinite(ey) and ey <= TOL[synth.BF16], ey
    assert np.isfinite(eh) and eh <= TOL[synth.BF16], eh


@pytest.mark.parametrize("shape,seed,a_scale", [
    # 128-token chunks of 128-wide heads, B in groups of heads, C per head;
    # few items, so the prepass and segments run too
    (F(2, 600, 8, 128, 128, 2, 8, 128, synth.BF16, "all"), 34, 1.0),
    (F(1, 1000, 4, 128, 128, 1, 4, 128, synth.BF16, "half"), 35, 1.0),
    (F(2, 129, 2, 128, 128, 1, 2, 128, synth.BF16, "all"), 37, 1.0),
    # chunks decaying past the scaled form's range: left to the per-head body
    (F(2, 700, 8, 128, 128, 2, 8, 128, synth.BF16, "all"), 36, 30.0),
    (F(1, 900, 6, 128, 128, 3, 6, 128, synth.BF16, "all"), 38, 3.0),
])
def test_fwd_fused_wide_heads(shape, seed, a_scale, monkeypatch):
    """The one-pass kernel with one 128-wide head per item (the Llama-3-8B
    hybrid's head shape) matches the oracle."""
    set_form(monkeypatch, "fused")
    d = S.make_dims(shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate,
                    shape.ngroups_b, shape.ngroups_c)
    names = [S.ssd_fwd_stage_name(d, 128, i) for i in range(S.ssd_fwd_num_stages(d, 128))]
    assert names[-2:] == ["chunk_fused_hb", "chunk_scan_flagged"], names
    check_fwd_scaled_A(shape, seed, a_scale)


def test_fwd_fused_wide_heads_matches_two_pass(monkeypatch):
    shape = F(2, 1000, 8, 128, 128, 2, 8, 128, synth.BF16, "all")
    d = to_dev(synth.make_fwd_inputs(shape, 39), shape.io)
    monkeypatch.setenv("SSD_FUSED", "1")
    y1, h1 = run_fwd(d, 128)
    monkeypatch.setenv("SSD_FUSED", "0")
    y2, h2 = run_fwd(d, 128)
    assert (y1.float() - y2.float()).abs().max() / y2.float().abs().max() < 1e-2
    assert (h1 - h2).abs().max() / h2.abs().max() < 1e-2


def test_fwd_fused_matches_two_pass(monkeypatch):
    """The one-pass kernel and the two-pass head-pair kernels agree within the
    tolerance on the same inputs (both are compared with the oracle elsewhere)."""
    shape = F(2, 1500, 6, 64, 128, 1, 1, 256, synth.BF16, "all")
    d = to_dev(synth.make_fwd_inputs(shape, 33), shape.io)
    monkeypatch.setenv("SSD_FUSED", "1")
    y1, h1 = run_fwd(d, 256)
    monkeypatch.setenv("SSD_FUSED", "0")
    y2, h2 = run_fwd(d, 256)
    assert (y1.float() - y2.float()).abs().max() / y2.float().abs().max() < 1e-2
    assert (h1 - h2).abs().max() / h2.abs().max() < 1e-2


def test_fwd_tc_without_softplus_and_D():
    check_fwd(F(1, 300, 2, 64, 128, 1, 1, 256, synth.BF16, "all"), 41, dt_softplus=False,
              D_none=True)


def test_fwd_pair_form_without_softplus_and_D(monkeypatch):
    """The head-pair chunk scan (forced) with dt used as given and no D."""
    monkeypatch.setenv("SSD_CHUNK_SCAN", "pair")
    shape = F(2, 700, 5, 64, 128, 1, 1, 256, synth.BF16, "all")
    d = S.make_dims(shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate,
                    dt_softplus=False)
    assert "chunk_scan_hb" in [S.ssd_fwd_stage_name(d, 256, i)
                               for i in range(S.ssd_fwd_num_stages(d, 256))]
    check_fwd(shape, 43, dt_softplus=False, D_none=True)


def test_fwd_f32_without_softplus_and_D():
    check_fwd(F(1, 130, 2, 32, 32, 1, 1, 64, synth.F32, "all"), 42, dt_softplus=False,
              D_none=True)


def test_fwd_stage_path_matches_dtype():
    d = S.make_dims(8, 2048, 80, 64, 128)
    assert [S.ssd_fwd_stage_name(d, 256, i) for i in range(S.ssd_fwd_num_stages(d, 256))] == \
        ["chunk_fused_prepass", "chunk_fused_hb", "chunk_scan_flagged"]
    assert S.ssd_fwd_stage_name(d, 128, 1) == "chunk_scan_hl"


# ---------------------------------------------------------------- full sizes
@pytest.mark.parametrize("name", ["mamba2_2p7b", "long_16k", "hybrid_llama3_8b"])
def test_fwd_full_size(name):
    """The full workloads, in the launch configuration the benchmark times,
    element by element over every (b, h) pair."""
    shape = synth.WORKLOADS[name]
    check_fwd(shape, synth.WORKLOAD_SEEDS[name])


def test_fwd_split_with_carried_state_matches_whole():
    """A prompt processed in two calls, the second starting from the first's
    final state, gives the one-call result (sequential prefill)."""
    shape = F(2, 1000, 4, 64, 128, 1, 1, 256, synth.BF16, "all")
    inp = synth.make_fwd_inputs(shape, 51)
    d = to_dev(inp, shape.io)
    y, hf = run_fwd(d, 256)
    T1 = 512
    part = lambda k, sl: d[k][:, sl].contiguous()
    d1 = dict(d, x=part("x", slice(0, T1)), dt=part("dt", slice(0, T1)), B=part("B", slice(0, T1)),
              C=part("C", slice(0, T1)))
    y1, h1 = run_fwd(d1, 256)
    d2 = dict(d, x=part("x", slice(T1, None)), dt=part("dt", slice(T1, None)),
              B=part("B", slice(T1, None)), C=part("C", slice(T1, None)), h0=h1)
    y2, h2 = run_fwd(d2, 256)
    ycat = torch.cat([y1, y2], dim=1).float()
    assert (ycat - y.float()).abs().max() / y.float().abs().max() < 1e-2
    assert (h2 - hf).abs().max() / hf.abs().max() < 1e-2


def test_fwd_deterministic():
    shape = F(1, 700, 4, 64, 128, 1, 1, 256, synth.BF16, "all")
    d = to_dev(synth.make_fwd_inputs(shape, 52), shape.io)
    y1, h1 = run_fwd(d, 256)
    y2, h2 = run_fwd(d, 256)
    assert torch.equal(y1, y2) and torch.equal(h1, h2)


@pytest.mark.parametrize("shape,seed", [
    (F(2, 700, 4, 64, 128, 1, 1, 256, synth.BF16, "all"), 53),     # two tensor-core kernels
    (F(1, 2000, 2, 64, 128, 1, 1, 128, synth.BF16, "all"), 54),    # segmented state pass (3 kernels)
    (F(1, 300, 4, 64, 64, 1, 1, 64, synth.F32, "all"), 55),        # float32 path (4 kernels)
])
def test_fwd_graph_replay_equals_eager(shape, seed):
    """ssd_fwd captured in a CUDA graph and replayed twice gives the eager result
    bit for bit: every step of the call is enqueued on the caller's stream."""
    d = to_dev(synth.make_fwd_inputs(shape, seed), shape.io)
    y_ref, h_ref = run_fwd(d, shape.chunk)
    b, T, H, P = d["x"].shape
    dims = S.dims_of(d["x"], d["B"], d["C"])
    ws = S.workspace_for(dims, shape.chunk)
    y = torch.empty_like(d["x"])
    hf = torch.empty((b, H, d["B"].shape[3], P), device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        S.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"], shape.chunk, y, hf, ws,
                  stream=stream)  # warm-up: one-time function attributes outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        S.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"], shape.chunk, y, hf, ws,
                  stream=stream)
    for _ in range(2):
        y.fill_(float("nan"))
        hf.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        S.ssd_check_device_error()
        assert torch.equal(y, y_ref) and torch.equal(hf, h_ref)


def test_fwd_head_pair_path_graph_and_serial_launch_agree(monkeypatch):
    """The head-pair path with a split last wave (dt_decay, chunk_state_hb,
    state_fixup, chunk_scan_hb, each after the first a programmatic dependent
    of the one before): eager, replayed from a CUDA graph, and launched one
    after another (SSD_PDL=0) give the same bits."""
    monkeypatch.setenv("SSD_CHUNK_SCAN", "pair")
    shape = F(4, 1024, 80, 64, 128, 1, 1, 256, synth.BF16, "all")
    d = to_dev(synth.make_fwd_inputs(shape, 56), shape.io)
    y_ref, h_ref = run_fwd(d, 256)
    monkeypatch.setenv("SSD_PDL", "0")
    y_ser, h_ser = run_fwd(d, 256)
    assert torch.equal(y_ser, y_ref) and torch.equal(h_ser, h_ref)
    monkeypatch.delenv("SSD_PDL")
    b, T, H, P = d["x"].shape
    dims = S.dims_of(d["x"], d["B"], d["C"])
    ws = S.workspace_for(dims, 256)
    y = torch.empty_like(d["x"])
    hf = torch.empty((b, H, d["B"].shape[3], P), device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        S.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"], 256, y, hf, ws,
                  stream=stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        S.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"], 256, y, hf, ws,
                  stream=stream)
    for _ in range(2):
        y.fill_(float("nan"))
        hf.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        S.ssd_check_device_error()
        assert torch.equal(y, y_ref) and torch.equal(hf, h_ref)


def test_fwd_fused_graph_and_serial_launch_agree(monkeypatch):
    """The one-pass path with a prepass (dt -> prepass -> one-pass kernel ->
    flagged-head pass, each after the first a programmatic dependent of the
    one before): eager, replayed from a CUDA graph, and launched one after
    another (SSD_PDL=0) give the same bits; long-decay heads make the flagged
    pass do work."""
    set_form(monkeypatch, "fused")
    shape = F(4, 1024, 80, 64, 128, 1, 1, 256, synth.BF16, "all")
    inp = synth.make_fwd_inputs(shape, 57)
    inp["A"] = (inp["A"] * np.float32(12.0)).astype(np.float32)
    d = to_dev(inp, shape.io)
    y_ref, h_ref = run_fwd(d, 256)
    monkeypatch.setenv("SSD_PDL", "0")
    y_ser, h_ser = run_fwd(d, 256)
    assert torch.equal(y_ser, y_ref) and torch.equal(h_ser, h_ref)
    monkeypatch.delenv("SSD_PDL")
    b, T, H, P = d["x"].shape
    dims = S.dims_of(d["x"], d["B"], d["C"])
    ws = S.workspace_for(dims, 256)
    y = torch.empty_like(d["x"])
    hf = torch.empty((b, H, d["B"].shape[3], P), device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        S.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"], 256, y, hf, ws,
                  stream=stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        S.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"], 256, y, hf, ws,
                  stream=stream)
    for _ in range(2):
        y.fill_(float("nan"))
        hf.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        S.ssd_check_device_error()
        assert torch.equal(y, y_ref) and torch.equal(hf, h_ref)


def test_fwd_profiled_events():
    shape = synth.WORKLOADS["tiny_f32"]
    d = to_dev(synth.make_fwd_inputs(shape, 1000), shape.io)
    dims = S.dims_of(d["x"], d["B"], d["C"])
    ws = S.workspace_for(dims, 64)
    y = torch.empty_like(d["x"])
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(S.ssd_fwd_num_stages(dims, 64) + 1)]
    S.ssd_fwd_profiled(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], None, 64, y, None, ws, ev)
    torch.cuda.synchronize()
    for a, b in zip(ev[:-1], ev[1:]):
        assert a.elapsed_time(b) >= 0.0
    y2, _ = run_fwd(d, 64, with_final=False)
    assert torch.equal(y, y2)


# ---------------------------------------------------------------- multistep
def ms_device(inp, io, s):
    dt_io = torch.bfloat16 if io == synth.BF16 else torch.float32
    return dict(x=torch.from_numpy(inp["x"][s]).to(dt_io).cuda(),
                dt=torch.from_numpy(inp["dt"][s]).cuda(),
                B=torch.from_numpy(inp["B"][s]).to(dt_io).cuda(),
                C=torch.from_numpy(inp["C"][s]).to(dt_io).cuda(),
                j=torch.from_numpy(inp["j"][s]).cuda())


M = synth.MultistepShape


@pytest.mark.parametrize("shape,seed", [
    (M(3, 5, 4, 64, 128, 2, 4, synth.BF16, 1), 61),
    (M(2, 8, 4, 64, 128, 1, 1, synth.F32, 1), 62),
    (M(2, 1, 2, 32, 48, 1, 2, synth.F32, 1), 63),
    (M(2, 16, 2, 128, 256, 1, 1, synth.BF16, 1), 64),
    (M(1, 3, 3, 48, 16, 1, 3, synth.F32, 1), 65),
])
def test_multistep_small(shape, seed):
    inp = synth.make_multistep_inputs(shape, seed)
    d = ms_device(inp, shape.io, 0)
    A, D = torch.from_numpy(inp["A"]).cuda(), torch.from_numpy(inp["D"]).cuda()
    hc = torch.from_numpy(inp["h_cache"]).cuda()
    y, hj, hK = S.multistep(d["x"], d["dt"], A, d["B"], d["C"], D, hc, d["j"])
    S.ssd_check_device_error()
    yr, hjr, hKr = oracle.ssd_multistep(inp["x"][0], inp["dt"][0], inp["A"], inp["B"][0],
                                        inp["C"][0], inp["D"], inp["h_cache"], inp["j"][0])
    b, K, H, P = inp["x"][0].shape
    pairs = list(range(b * H))
    tol = TOL[shape.io]
    assert rel_err(y_pairs(y, pairs, H), yr) <= tol
    assert rel_err(h_pairs(hj, pairs, H), hjr) <= tol
    assert rel_err(h_pairs(hK, pairs, H), hKr) <= tol


def test_multistep_j_extremes_bit_exact():
    shape = M(4, 8, 4, 64, 128, 1, 1, synth.BF16, 1)
    inp = synth.make_multistep_inputs(shape, 66)
    d = ms_device(inp, shape.io, 0)
    A, D = torch.from_numpy(inp["A"]).cuda(), torch.from_numpy(inp["D"]).cuda()
    hc = torch.from_numpy(inp["h_cache"]).cuda()
    j = torch.tensor([0, 8, 0, 8], dtype=torch.int32, device="cuda")
    y, hj, hK = S.multistep(d["x"], d["dt"], A, d["B"], d["C"], D, hc, j)
    assert torch.equal(hj[0], hc[0]) and torch.equal(hj[2], hc[2])
    assert torch.equal(hj[1], hK[1]) and torch.equal(hj[3], hK[3])


def test_multistep_bad_j_reported():
    shape = M(2, 4, 2, 64, 128, 1, 1, synth.BF16, 1)
    inp = synth.make_multistep_inputs(shape, 67)
    d = ms_device(inp, shape.io, 0)
    A, D = torch.from_numpy(inp["A"]).cuda(), torch.from_numpy(inp["D"]).cuda()
    hc = torch.from_numpy(inp["h_cache"]).cuda()
    j = torch.tensor([1, 5], dtype=torch.int32, device="cuda")
    S.multistep(d["x"], d["dt"], A, d["B"], d["C"], D, hc, j)
    with pytest.raises(S.SsdError) as e:
        S.ssd_check_device_error()
    assert e.value.status == S.SSD_ERR_INVALID_ARG
    S.ssd_check_device_error()  # the word was cleared


def _chain(shape, inp, steps, graph: bool, hk_rows=None):
    """Speculative chain: each step continues from h_j (ping-pong buffers).
    With hk_rows (flat b * H + h indices), every step's h_K of those (b, h)
    pairs is also copied out, inside the graph, to a [steps, rows, N, P]
    buffer returned third."""
    dt_io = torch.bfloat16 if shape.io == synth.BF16 else torch.float32
    X = torch.from_numpy(inp["x"][:steps]).to(dt_io).cuda()
    DT = torch.from_numpy(inp["dt"][:steps]).cuda()
    BB = torch.from_numpy(inp["B"][:steps]).to(dt_io).cuda()
    CC = torch.from_numpy(inp["C"][:steps]).to(dt_io).cuda()
    J = torch.from_numpy(inp["j"][:steps]).cuda()
    A, D = torch.from_numpy(inp["A"]).cuda(), torch.from_numpy(inp["D"]).cuda()
    h0 = torch.from_numpy(inp["h_cache"]).cuda()
    bufs = [torch.empty_like(h0), torch.empty_like(h0)]
    hK = torch.empty_like(h0)
    Y = torch.empty_like(X)
    dims = S.dims_of(X[0], BB[0], CC[0])
    b, _, H, P = X[0].shape
    N = BB.shape[-1]
    rows = None if hk_rows is None else torch.tensor(hk_rows, dtype=torch.long, device="cuda")
    HK = None if rows is None else torch.empty((steps, len(hk_rows), N, P), device="cuda")

    def run():
        cur = h0
        for s in range(steps):
            nxt = bufs[s % 2]
            S.ssd_multistep(X[s], DT[s], A, BB[s], CC[s], D, cur, J[s], Y[s], nxt, hK, dims=dims)
            if rows is not None:
                torch.index_select(hK.view(b * H, N, P), 0, rows, out=HK[s])
            cur = nxt
        return cur

    out = run()
    torch.cuda.synchronize()
    if not graph:
        return (Y, out) if rows is None else (Y, out, HK)
    Y.fill_(float("nan"))
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        out = run()
    g.replay()
    torch.cuda.synchronize()
    return (Y, out) if rows is None else (Y, out, HK)


def test_multistep_chain_full_size_sampled():
    """The 1000-step speculative chain at the full decode shape, in the graph
    the benchmark replays; sampled (b, h) pairs (every 20th) follow the
    oracle's chain on every step: y of every step and h_K of every step (the
    state after all K drafts, which the next step does not read), and the
    state the chain ends in (h_j of the last step)."""
    shape = synth.WORKLOADS["multistep_k8"]
    steps = shape.steps
    inp = synth.make_multistep_inputs(shape, synth.WORKLOAD_SEEDS["multistep_k8"])
    b, K, H, P = inp["x"][0].shape
    pairs = list(range(0, b * H, 20))
    Y, h_last, HK = _chain(shape, inp, steps, graph=True, hk_rows=pairs)
    S.ssd_check_device_error()
    Yh = Y.float().cpu().numpy()
    HKh = HK.cpu().numpy()
    cache = inp["h_cache"].copy()
    worst_y = worst_k = 0.0
    for s in range(steps):
        yr, hjr, hkr = oracle.ssd_multistep(inp["x"][s], inp["dt"][s], inp["A"], inp["B"][s],
                                            inp["C"][s], inp["D"], cache, inp["j"][s],
                                            pairs=pairs)
        # the oracle continues from its own states (float32-rounded like the GPU's)
        for q, p in enumerate(pairs):
            cache[p // H, p % H] = hjr[q].astype(np.float32)
        ys = np.stack([Yh[s, p // H, :, p % H, :] for p in pairs]).astype(np.float64)
        worst_y = max(worst_y, rel_err(ys, yr))
        worst_k = max(worst_k, rel_err(HKh[s].astype(np.float64), hkr))
    assert worst_y <= 1e-2, worst_y
    assert worst_k <= 1e-2, worst_k
    assert rel_err(h_pairs(h_last, pairs, H), np.stack([cache[p // H, p % H] for p in pairs])) <= 1e-2


def test_multistep_graph_equals_eager():
    shape = M(4, 8, 8, 64, 128, 1, 1, synth.BF16, 20)
    inp = synth.make_multistep_inputs(shape, 68)
    Y1, h1 = _chain(shape, inp, 20, graph=False)
    Y2, h2 = _chain(shape, inp, 20, graph=True)
    assert torch.equal(Y1, Y2) and torch.equal(h1, h2)
