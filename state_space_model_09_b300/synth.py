"""Seeded synthetic inputs for the SSD layer and the multi-step decode.

This module draws random numbers and nothing else: it holds none of the
layer's arithmetic (no softplus of dt, no decay, no recurrence).  Both the GPU
tests and the fp64 oracle consume exactly the arrays returned here, so the two
sides see the same bits.

Value recipe (the layer-level distributions the Mamba-2 2.7B workload uses):

* x ~ N(0, 1); B, C ~ N(0, 1/N)  (second parameter = variance);
* dt_raw = bias_h + r with r ~ N(0, 0.1); bias_h is chosen so that at r = 0
  the softplus'd step dt0_h is log-uniform in [1e-3, 1e-1], i.e.
  bias_h = dt0_h + log(-expm1(-dt0_h)) (the inverse of softplus);
* A_h = -exp(U[log 1, log 16]);  D_h ~ N(0, 1);
* initial states h0 ~ N(0, 0.1) where a workload asks for them.

x, B and C are rounded (round-to-nearest-even) to the I/O dtype before they
are returned, and returned as float32 arrays holding exactly those values;
dt_raw, A, D and the states are float32.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

F32 = 0
BF16 = 1


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even), as float32.

    Works on the bit pattern: add 0x7FFF plus the lowest kept bit, then clear
    the low 16 bits.  Finite inputs cannot overflow 32 bits this way."""
    out = np.array(a, dtype=np.float32, copy=True, order="C")
    u = out.view(np.uint32)
    step = 1 << 24
    flat = u.reshape(-1)
    for s in range(0, flat.size, step):
        blk = flat[s:s + step]
        lsb = (blk >> 16) & 1
        blk += np.uint32(0x7FFF) + lsb
        blk &= np.uint32(0xFFFF0000)
    return out


@dataclasses.dataclass(frozen=True)
class FwdShape:
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups_b: int = 1
    ngroups_c: int = 1
    chunk: int = 64
    io: int = F32
    h0: str = "zero"          # "zero" | "half" (first half of the batch random) | "all"

    @property
    def tok_heads(self) -> int:
        return self.batch * self.seqlen * self.nheads


@dataclasses.dataclass(frozen=True)
class MultistepShape:
    batch: int
    K: int
    nheads: int
    headdim: int
    dstate: int
    ngroups_b: int = 1
    ngroups_c: int = 1
    io: int = BF16
    steps: int = 1


# The five workloads: a tiny fp32 case, a Mamba-2 2.7B layer, a 16K-token
# sequence, a Llama-3-8B-shaped hybrid layer with grouped B, and the
# speculative multi-step verification decode.
WORKLOADS = {
    "tiny_f32": FwdShape(1, 256, 4, 64, 64, 1, 1, 64, F32, "zero"),
    "mamba2_2p7b": FwdShape(8, 2048, 80, 64, 128, 1, 1, 256, BF16, "half"),
    "long_16k": FwdShape(1, 16384, 80, 64, 128, 1, 1, 256, BF16, "zero"),
    "hybrid_llama3_8b": FwdShape(4, 4096, 32, 128, 128, 8, 32, 128, BF16, "zero"),
    "multistep_k8": MultistepShape(16, 8, 80, 64, 128, 1, 1, BF16, 1000),
}
WORKLOAD_SEEDS = {
    "tiny_f32": 1000,
    "mamba2_2p7b": 1001,
    "long_16k": 1002,
    "hybrid_llama3_8b": 1003,
    "multistep_k8": 1004,
}


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _normal(rng, shape, var: float) -> np.ndarray:
    out = rng.standard_normal(size=shape, dtype=np.float32)
    if var != 1.0:
        out *= np.float32(math.sqrt(var))
    return out


def head_params(rng, nheads: int):
    """Per-head A, D and dt bias (float32)."""
    log_dt0 = rng.uniform(math.log(1e-3), math.log(1e-1), size=nheads)
    dt0 = np.exp(log_dt0)
    bias = dt0 + np.log(-np.expm1(-dt0))
    A = -np.exp(rng.uniform(math.log(1.0), math.log(16.0), size=nheads))
    D = rng.standard_normal(size=nheads)
    return A.astype(np.float32), D.astype(np.float32), bias.astype(np.float32)


def _io_round(a: np.ndarray, io: int) -> np.ndarray:
    return round_to_bf16(a) if io == BF16 else a


def make_fwd_inputs(shape: FwdShape, seed: int):
    """Inputs of one prefill call, as a dict of float32 numpy arrays.

    Layouts: x [b,T,H,P]; dt [b,T,H]; B [b,T,G_B,N]; C [b,T,G_C,N]; A, D [H];
    h0 [b,H,N,P] or None.
    """
    s = shape
    rng = _rng(seed)
    A, D, bias = head_params(rng, s.nheads)
    x = _io_round(_normal(rng, (s.batch, s.seqlen, s.nheads, s.headdim), 1.0), s.io)
    B = _io_round(_normal(rng, (s.batch, s.seqlen, s.ngroups_b, s.dstate), 1.0 / s.dstate), s.io)
    C = _io_round(_normal(rng, (s.batch, s.seqlen, s.ngroups_c, s.dstate), 1.0 / s.dstate), s.io)
    r = _normal(rng, (s.batch, s.seqlen, s.nheads), 0.1)
    dt = (r + bias[None, None, :]).astype(np.float32)
    h0: Optional[np.ndarray] = None
    if s.h0 != "zero":
        h0 = _normal(rng, (s.batch, s.nheads, s.dstate, s.headdim), 0.1)
        if s.h0 == "half":
            h0[s.batch // 2:] = 0.0
    return dict(x=x, dt=dt, A=A, B=B, C=C, D=D, h0=h0)


def make_multistep_inputs(shape: MultistepShape, seed: int, steps: Optional[int] = None):
    """Inputs of a chain of multi-step decode calls.

    Per step s: x [b,K,H,P], dt [b,K,H], B [b,K,G_B,N], C [b,K,G_C,N] and the
    accepted count j [b] in 0..K (int32), drawn up front; plus the first cached
    state h_cache [b,H,N,P] ~ N(0, 0.1) and per-head A, D.  Arrays carry a
    leading step axis.
    """
    s = shape
    steps = s.steps if steps is None else steps
    rng = _rng(seed)
    A, D, bias = head_params(rng, s.nheads)
    h_cache = _normal(rng, (s.batch, s.nheads, s.dstate, s.headdim), 0.1)
    j = rng.integers(0, s.K + 1, size=(steps, s.batch), dtype=np.int64).astype(np.int32)
    x = _io_round(_normal(rng, (steps, s.batch, s.K, s.nheads, s.headdim), 1.0), s.io)
    B = _io_round(_normal(rng, (steps, s.batch, s.K, s.ngroups_b, s.dstate), 1.0 / s.dstate), s.io)
    C = _io_round(_normal(rng, (steps, s.batch, s.K, s.ngroups_c, s.dstate), 1.0 / s.dstate), s.io)
    r = _normal(rng, (steps, s.batch, s.K, s.nheads), 0.1)
    dt = (r + bias[None, None, None, :]).astype(np.float32)
    return dict(x=x, dt=dt, A=A, B=B, C=C, D=D, h_cache=h_cache, j=j)
