"""Pins of the fp64 oracle to facts other than itself (CPU only).

The pages print no worked example, so every pin is an identity the method
fixes, a closed form, or brute force on tiny inputs:

* duality: the recurrence equals multiplication by the masked T x T matrix
  M = L o (C B^T) (cloud.tencent page on Mamba-2, section "研究贡献" and
  "SSD算法": linear recurrence vs quadratic naive matmul);
* A = 0 reduces to causal linear attention (csdn page on "Mamba in the Llama",
  section "从 Transformer 到 Mamba": a linear RNN is linear attention);
* the chunked block decomposition is exact for every block size (Mamba-2
  page, section "SSD算法", the four coloured steps);
* a sequence split with its state carried equals the whole run (Mamba-2
  page, section on context parallelism; Falcon Mamba page, sequential
  prefill);
* closed forms: geometric series for N = P = 1, x = 0, B = 0, C = 0;
* MultiStep: K = 1, j = 0, j = K, equality with the sequential run, and a
  chain of speculative steps equals one run over the accepted tokens
  ("Mamba in the Llama", section 推测解码, MultiStep / FirstConflict).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from state_space_model_09_b300 import synth

TOL = 1e-12
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rel(a, b):
    return float(np.abs(np.asarray(a) - np.asarray(b)).max() / max(np.abs(np.asarray(b)).max(), 1e-300))


def small_inputs(seed, b=2, T=37, H=4, P=3, N=5, GB=2, GC=4, h0=True, io=synth.F32):
    shape = synth.FwdShape(b, T, H, P, N, GB, GC, 8, io, "all" if h0 else "zero")
    return synth.make_fwd_inputs(shape, seed)


def softplus_ref(z):
    # np.logaddexp(0, z) = log(1 + e^z), evaluated without overflow
    return np.logaddexp(0.0, z.astype(np.float64))


def quadratic_form(inp, dt_softplus=True):
    """Brute force: y = (L o C B^T) x + diag(exp(cs)) C h0 + D x with the
    full T x T lower-triangular L[t, s] = exp(cs_t - cs_s)."""
    x, B, C = (inp[k].astype(np.float64) for k in ("x", "B", "C"))
    b, T, H, P = x.shape
    GB, GC = B.shape[2], C.shape[2]
    dt = softplus_ref(inp["dt"]) if dt_softplus else inp["dt"].astype(np.float64)
    A = inp["A"].astype(np.float64)
    D = inp["D"].astype(np.float64) if inp["D"] is not None else np.zeros(H)
    h0 = inp["h0"]
    ys, hs = [], []
    for bi in range(b):
        for h in range(H):
            Bm = B[bi, :, h // (H // GB), :]          # [T, N]
            Cm = C[bi, :, h // (H // GC), :]
            cs = np.cumsum(dt[bi, :, h] * A[h])       # inclusive
            seg = cs[:, None] - cs[None, :]
            L = np.where(np.tril(np.ones((T, T), dtype=bool)), np.exp(np.minimum(seg, 0.0)), 0.0)
            M = L * (Cm @ Bm.T)
            y = M @ x[bi, :, h, :] + D[h] * x[bi, :, h, :]
            hT = (np.exp(cs[-1] - cs)[:, None] * Bm).T @ x[bi, :, h, :]
            if h0 is not None:
                H0 = h0[bi, h].astype(np.float64)
                y = y + np.exp(cs)[:, None] * (Cm @ H0)
                hT = hT + math.exp(cs[-1]) * H0
            ys.append(y)
            hs.append(hT)
    return np.stack(ys), np.stack(hs)


def run_seq(inp, **kw):
    return oracle.ssd_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"], **kw)


@pytest.mark.parametrize("seed,h0,GB,GC", [(1, True, 2, 4), (2, False, 1, 1), (3, True, 4, 2)])
def test_quadratic_form_duality(seed, h0, GB, GC):
    inp = small_inputs(seed, h0=h0, GB=GB, GC=GC)
    y, h = run_seq(inp)
    yq, hq = quadratic_form(inp)
    assert rel(y, yq) < TOL
    assert rel(h, hq) < TOL


def test_quadratic_form_without_softplus():
    inp = small_inputs(4)
    inp["dt"] = np.abs(inp["dt"]) * np.float32(0.05)
    y, h = run_seq(inp, dt_softplus=False)
    yq, hq = quadratic_form(inp, dt_softplus=False)
    assert rel(y, yq) < TOL and rel(h, hq) < TOL


def test_softplus_matches_its_inverse():
    """softplus(log(expm1(d))) = d: feeding the inverse-softplus of a positive
    step with the flag on equals feeding the step itself with the flag off."""
    inp = small_inputs(5)
    d = np.random.default_rng(0).uniform(1e-3, 0.5, size=inp["dt"].shape)
    raw = np.log(np.expm1(d))
    inp_raw = dict(inp, dt=raw.astype(np.float32))
    inp_pos = dict(inp, dt=softplus_ref(raw.astype(np.float32)).astype(np.float32))
    y1, h1 = run_seq(inp_raw, dt_softplus=True)
    # the flag-off run sees dt rounded to float32, so allow float32 rounding
    y2, h2 = run_seq(inp_pos, dt_softplus=False)
    assert rel(y1, y2) < 1e-6 and rel(h1, h2) < 1e-6
    # large arguments: softplus(z) -> z above the threshold (exact to 1e-9)
    big = dict(inp, dt=np.full_like(inp["dt"], 25.0), A=np.full_like(inp["A"], -0.01))
    y3, h3 = run_seq(big, dt_softplus=True)
    big_off = dict(big, dt=np.full_like(inp["dt"], 25.0))
    y4, h4 = run_seq(big_off, dt_softplus=False)
    assert rel(y3, y4) < 1e-9


def test_zero_A_is_causal_linear_attention():
    inp = small_inputs(6, T=23)
    inp["A"] = np.zeros_like(inp["A"])
    y, h = run_seq(inp)
    x, B, C = (inp[k].astype(np.float64) for k in ("x", "B", "C"))
    b, T, H, P = x.shape
    GB, GC = B.shape[2], C.shape[2]
    q = 0
    for bi in range(b):
        for hh in range(H):
            H0 = inp["h0"][bi, hh].astype(np.float64)
            for t in range(T):
                Ct = C[bi, t, hh // (H // GC)]
                acc = Ct @ H0 + inp["D"][hh] * x[bi, t, hh]
                for s in range(t + 1):
                    acc = acc + (Ct @ B[bi, s, hh // (H // GB)]) * x[bi, s, hh]
                assert np.abs(acc - y[q, t]).max() <= TOL * max(1.0, np.abs(acc).max())
            q += 1


@pytest.mark.parametrize("Q", [1, 4, 7, 16, 64, 100, 1000])
def test_chunk_size_invariance(Q):
    inp = small_inputs(7, T=96, P=4, N=6)
    y, h = run_seq(inp)
    yc, hc = oracle.ssd_chunked(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                                inp["h0"], chunk=Q)
    assert rel(yc, y) < TOL
    assert rel(hc, h) < TOL


def test_chunked_matches_quadratic_form_directly():
    inp = small_inputs(8, T=50)
    yc, hc = oracle.ssd_chunked(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                                inp["h0"], chunk=16)
    yq, hq = quadratic_form(inp)
    assert rel(yc, yq) < TOL and rel(hc, hq) < TOL


@pytest.mark.parametrize("T1", [1, 17, 40])
def test_split_with_carried_state(T1):
    inp = small_inputs(9, T=41)
    b, T, H, P = inp["x"].shape
    N = inp["B"].shape[3]
    y, h = run_seq(inp)
    first = {k: (v[:, :T1] if k in ("x", "dt", "B", "C") else v) for k, v in inp.items()}
    y1, h1 = run_seq(first)
    second = {k: (v[:, T1:] if k in ("x", "dt", "B", "C") else v) for k, v in inp.items()}
    second["h0"] = h1.reshape(b, H, N, P).astype(np.float32)
    # the carried state is rounded to float32 on the way back in
    y2, h2 = run_seq(second)
    assert rel(np.concatenate([y1, y2], axis=1), y) < 1e-6
    assert rel(h2, h) < 1e-6


def test_geometric_series_closed_form():
    """N = P = 1, constant a, B, x:  h_t = a^t h0 + B x (1 - a^t) / (1 - a)."""
    T = 50
    dtv, Av, Bv, xv, Cv, Dv, h0v = 0.3, -0.7, 0.8, -1.25, 0.6, 0.4, 2.0
    inp = dict(x=np.full((1, T, 1, 1), xv, np.float32), dt=np.full((1, T, 1), dtv, np.float32),
               A=np.array([Av], np.float32), B=np.full((1, T, 1, 1), Bv, np.float32),
               C=np.full((1, T, 1, 1), Cv, np.float32), D=np.array([Dv], np.float32),
               h0=np.full((1, 1, 1, 1), h0v, np.float32))
    y, h = run_seq(inp, dt_softplus=False)
    a = math.exp(np.float32(dtv) * np.float64(np.float32(Av)))
    f = lambda v: float(np.float32(v))
    for t in range(1, T + 1):
        ht = a ** t * f(h0v) + f(Bv) * f(xv) * (1 - a ** t) / (1 - a)
        yt = f(Cv) * ht + f(Dv) * f(xv)
        assert abs(y[0, t - 1, 0] - yt) <= 1e-13 * max(1.0, abs(yt))
    assert abs(h[0, 0, 0] - (a ** T * f(h0v) + f(Bv) * f(xv) * (1 - a ** T) / (1 - a))) < 1e-13


def test_zero_input_decays_initial_state():
    inp = small_inputs(10, T=30)
    inp["x"] = np.zeros_like(inp["x"])
    y, h = run_seq(inp)
    b, T, H, P = inp["x"].shape
    GC = inp["C"].shape[2]
    dt = softplus_ref(inp["dt"])
    q = 0
    for bi in range(b):
        for hh in range(H):
            cs = np.cumsum(dt[bi, :, hh] * np.float64(inp["A"][hh]))
            H0 = inp["h0"][bi, hh].astype(np.float64)
            assert rel(h[q], math.exp(cs[-1]) * H0) < TOL
            Cm = inp["C"][bi, :, hh // (H // GC)].astype(np.float64)
            assert rel(y[q], np.exp(cs)[:, None] * (Cm @ H0)) < TOL
            q += 1


def test_zero_B_and_zero_C():
    inp = small_inputs(11, T=20)
    b, T, H, P = inp["x"].shape
    xb = inp["x"].astype(np.float64)
    # C = 0: y = D x whatever the state
    y, _ = run_seq(dict(inp, C=np.zeros_like(inp["C"])))
    ref = np.stack([inp["D"][hh] * xb[bi, :, hh] for bi in range(b) for hh in range(H)])
    assert rel(y, ref) < TOL
    # B = 0 and h0 = 0: the state stays zero, y = D x
    y, h = run_seq(dict(inp, B=np.zeros_like(inp["B"]), h0=None))
    assert rel(y, ref) < TOL and np.abs(h).max() == 0.0


def test_dyadic_example_exact():
    """A = 0 and dyadic values make every operation exact in binary, so the
    recurrence can be evaluated by hand: h_t = h0 + sum_{s<=t} B_s x_s^T and
    y_t = C_t^T h_t + D x_t, with N = P = 2 and T = 3."""
    x = np.array([[1.0, -2.0], [0.5, 0.25], [-1.0, 4.0]])
    B = np.array([[1.0, 0.0], [0.5, -1.0], [2.0, 0.25]])
    C = np.array([[0.0, 1.0], [1.0, 1.0], [-0.5, 2.0]])
    h0 = np.array([[1.0, 2.0], [3.0, 4.0]])
    D = 0.5
    inp = dict(x=x.reshape(1, 3, 1, 2).astype(np.float32), dt=np.ones((1, 3, 1), np.float32),
               A=np.zeros(1, np.float32), B=B.reshape(1, 3, 1, 2).astype(np.float32),
               C=C.reshape(1, 3, 1, 2).astype(np.float32), D=np.array([D], np.float32),
               h0=h0.reshape(1, 1, 2, 2).astype(np.float32))
    y, h = run_seq(inp, dt_softplus=False)
    # by hand: h1 = [[2, 0], [3, 4]]; y1 = [3, 4] + [0.5, -1] = [3.5, 3]
    #          h2 = [[2.25, 0.125], [2.5, 3.75]]; y2 = [4.75, 3.875] + [0.25, 0.125]
    #          h3 = [[0.25, 8.125], [2.25, 4.75]]; y3 = [4.375, 5.4375] + [-0.5, 2]
    assert np.array_equal(h[0], [[0.25, 8.125], [2.25, 4.75]])
    assert np.array_equal(y[0], [[3.5, 3.0], [5.0, 4.0], [3.875, 7.4375]])


def test_golden_regression():
    """Outputs stored by tests/golden/make_golden.py (which calls only the
    oracle) still come out the same: guards the oracle against drift."""
    with open(os.path.join(GOLDEN, "oracle_tiny.json")) as f:
        g = json.load(f)
    shape = synth.FwdShape(**g["shape"])
    inp = synth.make_fwd_inputs(shape, g["seed"])
    y, h = run_seq(inp)
    assert rel(y[:, :g["T_stored"]], np.array(g["y_head"])) < TOL
    assert rel(h, np.array(g["h_final"])) < TOL


# ---------------------------------------------------------------- multistep

def ms_inputs(seed, b=3, K=5, H=4, P=3, N=5, GB=2, GC=4, steps=1):
    shape = synth.MultistepShape(b, K, H, P, N, GB, GC, synth.F32, steps)
    return synth.make_multistep_inputs(shape, seed)


def run_ms(inp, s, h_cache, j):
    return oracle.ssd_multistep(inp["x"][s], inp["dt"][s], inp["A"], inp["B"][s], inp["C"][s],
                                inp["D"], h_cache, j)


def test_multistep_equals_sequential_run():
    inp = ms_inputs(20)
    b, K, H, P = inp["x"][0].shape
    N = inp["B"].shape[-1]
    y, hj, hK = run_ms(inp, 0, inp["h_cache"], inp["j"][0])
    ys, hs = oracle.ssd_seq(inp["x"][0], inp["dt"][0], inp["A"], inp["B"][0], inp["C"][0],
                            inp["D"], inp["h_cache"])
    assert rel(y, ys) < TOL and rel(hK, hs) < TOL
    # h_j is the sequential state after the first j tokens of this call
    for bi in range(b):
        jb = int(inp["j"][0][bi])
        for hh in range(H):
            q = bi * H + hh
            if jb == 0:
                ref = inp["h_cache"][bi, hh].astype(np.float64)
            else:
                _, hpre = oracle.ssd_seq(inp["x"][0][bi:bi + 1, :jb], inp["dt"][0][bi:bi + 1, :jb],
                                         inp["A"], inp["B"][0][bi:bi + 1, :jb],
                                         inp["C"][0][bi:bi + 1, :jb], inp["D"],
                                         inp["h_cache"][bi:bi + 1], pairs=[hh])
                ref = hpre[0]
            assert rel(hj[q], ref) < TOL


def test_multistep_j_extremes_and_K1():
    inp = ms_inputs(21)
    b = inp["x"].shape[1]
    K = inp["x"].shape[2]
    y, hj, hK = run_ms(inp, 0, inp["h_cache"], np.zeros(b, np.int32))
    H = inp["x"].shape[3]
    assert np.array_equal(hj, inp["h_cache"].astype(np.float64).reshape(b * H, *hj.shape[1:]))
    y, hj, hK = run_ms(inp, 0, inp["h_cache"], np.full(b, K, np.int32))
    assert np.array_equal(hj, hK)
    # K = 1 is one step of the recurrence, written out here directly
    one = {k: (v[:, :, :1] if k in ("x", "dt", "B", "C") else v) for k, v in inp.items()}
    y1, hj1, hK1 = run_ms(one, 0, inp["h_cache"], np.ones(b, np.int32))
    x, B, C = (one[k][0].astype(np.float64) for k in ("x", "B", "C"))
    GB, GC = B.shape[2], C.shape[2]
    for bi in range(b):
        for hh in range(H):
            a = math.exp(softplus_ref(one["dt"][0][bi, 0, hh:hh + 1])[0] * np.float64(inp["A"][hh]))
            hn = a * inp["h_cache"][bi, hh].astype(np.float64) + np.outer(B[bi, 0, hh // (H // GB)], x[bi, 0, hh])
            yn = C[bi, 0, hh // (H // GC)] @ hn + inp["D"][hh] * x[bi, 0, hh]
            assert rel(hK1[bi * H + hh], hn) < TOL and rel(y1[bi * H + hh, 0], yn) < TOL


def test_multistep_rejects_bad_j():
    inp = ms_inputs(22)
    b, K = inp["x"].shape[1], inp["x"].shape[2]
    with pytest.raises(ValueError):
        run_ms(inp, 0, inp["h_cache"], np.full(b, K + 1, np.int32))


def test_speculative_chain_equals_run_over_accepted_tokens():
    """Each step continues from h_j (= h_K when all K drafts were accepted);
    the chain equals one sequential run over every step's accepted tokens."""
    steps = 12
    inp = ms_inputs(23, steps=steps)
    b, K, H, P = inp["x"][0].shape
    N = inp["B"].shape[-1]
    cache = inp["h_cache"].copy()
    ys = [[] for _ in range(b)]
    for s in range(steps):
        y, hj, hK = run_ms(inp, s, cache, inp["j"][s])
        for bi in range(b):
            jb = int(inp["j"][s][bi])
            ys[bi].append(y.reshape(b, H, K, P)[bi, :, :jb])
        cache = hj.reshape(b, H, N, P).astype(np.float32)
    for bi in range(b):
        acc = [int(inp["j"][s][bi]) for s in range(steps)]
        if sum(acc) == 0:
            continue
        cat = lambda k: np.concatenate([inp[k][s][bi:bi + 1, :acc[s]] for s in range(steps)], axis=1)
        y_seq, h_seq = oracle.ssd_seq(cat("x"), cat("dt"), inp["A"], cat("B"), cat("C"), inp["D"],
                                      inp["h_cache"][bi:bi + 1])
        y_chain = np.concatenate(ys[bi], axis=1)          # [H, sum(acc), P]
        # the chain rounds its carried state to float32 at every step
        assert rel(y_chain, y_seq) < 1e-6
        assert rel(cache[bi], h_seq.reshape(H, N, P)) < 1e-6
