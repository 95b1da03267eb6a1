"""Fused verification with recompute (ssd_verify): the cache holds the state
before the previous call's drafts; one kernel advances it through the
accepted ones, stores the next cache and decodes the new drafts."""
import numpy as np
import pytest
import torch

import oracle
from state_space_model_09_b300 import ssd as S
from state_space_model_09_b300 import synth

pytestmark = pytest.mark.gpu

M = synth.MultistepShape
TOL = {synth.F32: 1e-4, synth.BF16: 1e-2}


def _steps(inp, io, s):
    dt_io = torch.bfloat16 if io == synth.BF16 else torch.float32
    return dict(x=torch.from_numpy(inp["x"][s]).to(dt_io).cuda(),
                dt=torch.from_numpy(inp["dt"][s]).cuda(),
                B=torch.from_numpy(inp["B"][s]).to(dt_io).cuda(),
                C=torch.from_numpy(inp["C"][s]).to(dt_io).cuda(),
                j=torch.from_numpy(inp["j"][s]).cuda())


@pytest.mark.parametrize("shape,seed", [
    (M(3, 8, 4, 64, 128, 1, 1, synth.BF16, 2), 71),   # the decode shape's specialised instance
    (M(2, 5, 4, 32, 64, 2, 4, synth.F32, 2), 72),     # groups, float32, K = 5
    (M(2, 12, 2, 128, 256, 1, 1, synth.BF16, 2), 77),  # 16-token instance, 128-column slices
    (M(2, 3, 4, 64, 64, 1, 2, synth.BF16, 2), 78),    # bf16, N = 64: the generic instance
])
def test_verify_matches_oracle(shape, seed):
    inp = synth.make_multistep_inputs(shape, seed, steps=2)
    prev, cur = _steps(inp, shape.io, 0), _steps(inp, shape.io, 1)
    jp = prev["j"].clone()
    jp[0] = 0
    jp[-1] = shape.K  # both extremes
    A, D = torch.from_numpy(inp["A"]).cuda(), torch.from_numpy(inp["D"]).cuda()
    h_cache = torch.from_numpy(inp["h_cache"]).cuda()
    y = torch.full_like(cur["x"], float("nan"))
    h_next = torch.full_like(h_cache, float("nan"))
    S.ssd_verify(prev["x"], prev["dt"], prev["B"], jp, cur["x"], cur["dt"], A, cur["B"],
                 cur["C"], D, h_cache, y, h_next)
    torch.cuda.synchronize()
    S.ssd_check_device_error()
    # oracle: h_next = state after the first jp tokens of the previous drafts,
    # y = the new drafts decoded from it
    b, H = shape.batch, shape.nheads
    pairs = list(range(b * H))
    f64 = lambda t: t.float().cpu().numpy().astype(np.float64)
    _, h_ref, _ = oracle.ssd_multistep(f64(prev["x"]), inp["dt"][0], inp["A"], f64(prev["B"]),
                                       f64(prev["B"]), inp["D"], inp["h_cache"],
                                       jp.cpu().numpy(), pairs=pairs)
    h_ref_full = h_ref.reshape(b, H, shape.dstate, shape.headdim)
    y_ref, _, _ = oracle.ssd_multistep(f64(cur["x"]), inp["dt"][1], inp["A"], f64(cur["B"]),
                                       f64(cur["C"]), inp["D"], h_ref_full,
                                       np.zeros(b, dtype=np.int32), pairs=pairs)
    hn = f64(h_next).reshape(b * H, shape.dstate, shape.headdim)
    yy = f64(y)
    ys = np.stack([yy[p // H, :, p % H, :] for p in pairs])
    tol = TOL[shape.io]
    assert np.abs(hn - h_ref).max() / np.abs(h_ref).max() <= tol
    assert np.abs(ys - y_ref).max() / np.abs(y_ref).max() <= tol


def test_verify_chain_equals_multistep_chain_bit_exact():
    """A chain of ssd_verify calls (cache = state before the previous drafts)
    reproduces a chain of ssd_multistep calls continuing from h_j, bit for
    bit: the recompute performs the same operations in the same order."""
    shape = M(4, 8, 6, 64, 128, 1, 1, synth.BF16, 12)
    steps = 12
    inp = synth.make_multistep_inputs(shape, 73, steps=steps)
    st = [_steps(inp, shape.io, s) for s in range(steps)]
    A, D = torch.from_numpy(inp["A"]).cuda(), torch.from_numpy(inp["D"]).cuda()
    h0 = torch.from_numpy(inp["h_cache"]).cuda()
    # multistep chain: states entering each step, outputs
    ms_h, ms_y = [h0.clone()], []
    hK = torch.empty_like(h0)
    for s in range(steps):
        y = torch.empty_like(st[s]["x"])
        hj = torch.empty_like(h0)
        S.ssd_multistep(st[s]["x"], st[s]["dt"], A, st[s]["B"], st[s]["C"], D, ms_h[-1],
                        st[s]["j"], y, hj, hK)
        ms_y.append(y)
        ms_h.append(hj)
    # verify chain
    cache = h0.clone()
    zero = torch.zeros_like(st[0]["j"])
    for s in range(steps):
        prev = st[s - 1] if s > 0 else st[0]
        jp = st[s - 1]["j"] if s > 0 else zero
        y = torch.empty_like(st[s]["x"])
        h_next = torch.empty_like(h0)
        S.ssd_verify(prev["x"], prev["dt"], prev["B"], jp, st[s]["x"], st[s]["dt"], A,
                     st[s]["B"], st[s]["C"], D, cache, y, h_next)
        torch.cuda.synchronize()
        assert torch.equal(h_next, ms_h[s]), s
        assert torch.equal(y, ms_y[s]), s
        cache = h_next
    S.ssd_check_device_error()


def test_verify_bad_j_prev_is_reported_and_row_untouched():
    shape = M(2, 4, 2, 64, 128, 1, 1, synth.BF16, 2)
    inp = synth.make_multistep_inputs(shape, 74, steps=2)
    prev, cur = _steps(inp, shape.io, 0), _steps(inp, shape.io, 1)
    jp = torch.tensor([1, 9], dtype=torch.int32, device="cuda")  # row 1 out of range
    A, D = torch.from_numpy(inp["A"]).cuda(), torch.from_numpy(inp["D"]).cuda()
    h_cache = torch.from_numpy(inp["h_cache"]).cuda()
    y = torch.full_like(cur["x"], float("nan"))
    h_next = torch.full_like(h_cache, float("nan"))
    S.ssd_verify(prev["x"], prev["dt"], prev["B"], jp, cur["x"], cur["dt"], A, cur["B"],
                 cur["C"], D, h_cache, y, h_next)
    with pytest.raises(S.SsdError) as e:
        S.ssd_check_device_error()
    assert e.value.status == S.SSD_ERR_INVALID_ARG
    assert torch.isfinite(y[0].float()).all() and torch.isfinite(h_next[0]).all()
    assert torch.isnan(y[1].float()).all() and torch.isnan(h_next[1]).all()


def test_draft_step_recompute_then_one_token():
    """Draft-model side: the first draft step of a round rolls the draft's
    cache through the j_prev accepted tokens of the previous round (8 slots)
    and decodes ONE new token, in one call (k_prev = 8, K = 1)."""
    prev_shape = M(3, 8, 4, 64, 128, 1, 1, synth.BF16, 1)
    new_shape = M(3, 1, 4, 64, 128, 1, 1, synth.BF16, 1)
    pin = synth.make_multistep_inputs(prev_shape, 75, steps=1)
    nin = synth.make_multistep_inputs(new_shape, 76, steps=1)
    prev, cur = _steps(pin, synth.BF16, 0), _steps(nin, synth.BF16, 0)
    jp = torch.tensor([0, 5, 8], dtype=torch.int32, device="cuda")
    A, D = torch.from_numpy(pin["A"]).cuda(), torch.from_numpy(pin["D"]).cuda()
    h_cache = torch.from_numpy(pin["h_cache"]).cuda()
    y = torch.full_like(cur["x"], float("nan"))
    h_next = torch.full_like(h_cache, float("nan"))
    S.ssd_verify(prev["x"], prev["dt"], prev["B"], jp, cur["x"], cur["dt"], A, cur["B"],
                 cur["C"], D, h_cache, y, h_next)
    torch.cuda.synchronize()
    S.ssd_check_device_error()
    b, H = 3, 4
    pairs = list(range(b * H))
    f64 = lambda t: t.float().cpu().numpy().astype(np.float64)
    _, h_ref, _ = oracle.ssd_multistep(f64(prev["x"]), pin["dt"][0], pin["A"], f64(prev["B"]),
                                       f64(prev["B"]), pin["D"], pin["h_cache"],
                                       jp.cpu().numpy(), pairs=pairs)
    y_ref, _, _ = oracle.ssd_multistep(f64(cur["x"]), nin["dt"][0], pin["A"], f64(cur["B"]),
                                       f64(cur["C"]), pin["D"], h_ref.reshape(b, H, 128, 64),
                                       np.zeros(b, dtype=np.int32), pairs=pairs)
    hn = f64(h_next).reshape(b * H, 128, 64)
    yy = f64(y)
    ys = np.stack([yy[p // H, :, p % H, :] for p in pairs])
    assert np.abs(hn - h_ref).max() / np.abs(h_ref).max() <= 1e-2
    assert np.abs(ys - y_ref).max() / np.abs(y_ref).max() <= 1e-2
