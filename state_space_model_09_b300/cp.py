"""Context parallelism over the sequence (Mamba-2 page, section
"序列并行的两种形式", context parallelism): the ranks of a process group each
hold one contiguous segment of every sequence, in rank order; every rank
computes its segment's outputs and final state, the states pass from rank to
rank, and each segment's outputs are corrected for the state it really starts
from.  See ssd_cp_workspace_size / ssd_cp_segment_decay / ssd_cp_correct in
ssd.h for the arithmetic; everything here is argument marshalling and the
all-gather (torch.distributed: NCCL on GPUs, gloo in the CPU tests).
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import ssd as S


def gather_segment_states(decay: torch.Tensor, h_final: torch.Tensor, group=None):
    """All-gather every rank's segment decay [b, H] and segment final state
    [b, H, N, P] into rank-ordered buffers [world, b, H] and
    [world, b, H, N, P] (communication only)."""
    world = dist.get_world_size(group)
    decays = torch.empty((world,) + tuple(decay.shape), dtype=decay.dtype, device=decay.device)
    finals = torch.empty((world,) + tuple(h_final.shape), dtype=h_final.dtype,
                         device=h_final.device)
    dist.all_gather(list(decays.unbind(0)), decay.contiguous(), group=group)
    dist.all_gather(list(finals.unbind(0)), h_final.contiguous(), group=group)
    return decays, finals


def context_parallel_forward(x, dt, A, B, C, D=None, h0=None, chunk: int = 256,
                             dt_softplus: bool = True, group=None):
    """This rank's segment of the layer with context parallelism: returns the
    segment's y and its true final state (the last rank's is the sequence's).
    x, dt, B, C are this rank's segment; h0 (the sequence's initial state) is
    used on rank 0 only.  Runs on torch's current stream."""
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    y, h_local = S.forward(x, dt, A, B, C, D, h0 if rank == 0 else None, chunk, dt_softplus)
    dims = S.dims_of(x, B, C, dt_softplus)
    ws = torch.empty(S.ssd_cp_workspace_size(dims), dtype=torch.uint8, device=x.device)
    b, _, H, _ = x.shape
    decay = torch.empty((b, H), dtype=torch.float32, device=x.device)
    S.ssd_cp_segment_decay(dt, A, decay, ws, dims)
    decays, finals = gather_segment_states(decay, h_local, group)
    h_final = torch.empty_like(h_local)
    S.ssd_cp_correct(world, rank, decays, finals, dt, A, C, y, h_final, ws, dims)
    return y, h_final
