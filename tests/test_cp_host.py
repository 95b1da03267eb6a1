"""Host protocol of context parallelism on gloo ranks (CPU): every rank holds
one segment of the sequence, computes that segment with the fp64 oracle from
a zero state (rank 0 from h0), and exchanges (segment decay, segment final
state) through cp.gather_segment_states.  Each rank then applies the
documented recurrence -- H_in(0) = 0, H_in(r + 1) = Lambda_r H_in(r) + F_r --
and correction -- y_t += exp(cs_t) C_t^T H_in, h_final = Lambda H_in + F --
here in numpy, and must reproduce the whole-sequence oracle: the gathered
buffers are rank-ordered and the protocol is complete.  (The GPU kernels that
do the combine and the correction are checked against the oracle in
test_gpu_cp.py.)"""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _softplus(z):
    return np.where(z > 20, z, np.log1p(np.exp(np.minimum(z, 20))))


def _rank_main(rank, world, port, cuts, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import oracle
    from state_space_model_09_b300 import cp, synth

    dist.init_process_group("gloo", rank=rank, world_size=world)
    shape = synth.FwdShape(2, 120, 3, 16, 8, 1, 3, 64, synth.F32, "all")
    inp = synth.make_fwd_inputs(shape, 77)
    bounds = [0] + list(cuts) + [shape.seqlen]
    sl = slice(bounds[rank], bounds[rank + 1])
    seg = {k: (v[:, sl] if k in ("x", "dt", "B", "C") else v) for k, v in inp.items()}
    b, H = shape.batch, shape.nheads
    pairs = list(range(b * H))
    y_loc, f_loc = oracle.ssd_seq(seg["x"], seg["dt"], seg["A"], seg["B"], seg["C"], seg["D"],
                                  seg["h0"] if rank == 0 else None, pairs=pairs)
    a = np.cumsum(_softplus(seg["dt"].astype(np.float64)) * inp["A"][None, None, :], axis=1)
    decay = np.exp(a[:, -1, :])  # [b, H]
    F = oracle.states_full(f_loc, b, H)  # [b, H, N, P]
    decays, finals = cp.gather_segment_states(torch.from_numpy(decay), torch.from_numpy(F))
    decays, finals = decays.numpy(), finals.numpy()
    assert decays.shape == (world, b, H) and finals.shape == (world,) + F.shape
    assert np.array_equal(decays[rank], decay) and np.array_equal(finals[rank], F)
    # the documented combine, then the correction of this segment
    Hin = np.zeros_like(F)
    for r in range(rank):
        Hin = decays[r][:, :, None, None] * Hin + finals[r]
    h_final = decay[:, :, None, None] * Hin + F
    y = oracle.to_full(y_loc, b, H).astype(np.float64)  # [b, t, H, P]
    g = np.arange(H) // (H // shape.ngroups_c)
    Cg = seg["C"][:, :, g, :].astype(np.float64)  # [b, t, H, N]
    y += np.exp(a)[..., None] * np.einsum("bthn,bhnp->bthp", Cg, Hin)
    # reference: the whole sequence, and the state at this segment's end
    cut = {k: (v[:, :bounds[rank + 1]] if k in ("x", "dt", "B", "C") else v)
           for k, v in inp.items()}
    yr, hr = oracle.ssd_seq(cut["x"], cut["dt"], cut["A"], cut["B"], cut["C"], cut["D"],
                            cut["h0"], pairs=pairs)
    yr = oracle.to_full(yr, b, H)[:, sl]
    hr = oracle.states_full(hr, b, H)
    ey = float(np.abs(y - yr).max() / np.abs(yr).max())
    eh = float(np.abs(h_final - hr).max() / np.abs(hr).max())
    q.put((rank, ey, eh))
    dist.destroy_process_group()


@pytest.mark.parametrize("world,cuts", [(2, (50,)), (3, (40, 41))])
def test_context_parallel_protocol_on_gloo_ranks(world, cuts):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, cuts, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert [r[0] for r in res] == list(range(world))
    for _, ey, eh in res:
        assert ey <= 1e-12 and eh <= 1e-12, (ey, eh)
