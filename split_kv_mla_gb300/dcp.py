"""Decode context parallelism (DCP): host plumbing around the two DCP entry
points of ``libmla.so``.

moonmath-ai/amd-kernels README, "MLA absorbed decode" and "Use / MLA decode":
under DCP rank ``cp_rank`` of ``cp_world`` holds the positions p of every request
with ``p % cp_world == cp_rank``; its decode call gets the global lengths
``glen`` and returns its share's output and base-2 LSE; after an all-to-all (or
all-gather) the shares are merged with ``mla_dcp_lse_merge_ranks``.

Nothing here computes attention: :func:`shard_page_table` lays out one rank's
page table (a serving stack normally writes each rank's cache that way from the
start; this builds the same view from a full table), :func:`all_gather_shares`
is the exchange step over ``torch.distributed`` (NCCL on GPUs, gloo on CPUs),
and :func:`dcp_decode_step` chains rank decode, exchange and merge, both
compute steps running in the library's kernels.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch
import torch.distributed as dist


def shard_page_table(seq_lens: torch.Tensor, kv_indices: torch.Tensor,
                     kv_indptr: torch.Tensor, cp_rank: int, cp_world: int):
    """Rank ``cp_rank``'s page table: request b keeps the slots of its positions
    p < seq_lens[b] with p % cp_world == cp_rank, in increasing p, so local key
    j is global position j * cp_world + cp_rank.  Returns
    (local_seq_lens, local_kv_indices, local_kv_indptr, glen), int32 tensors on
    the input's device; glen is a copy of seq_lens (the global lengths)."""
    if cp_world < 1 or not 0 <= cp_rank < cp_world:
        raise ValueError("need 0 <= cp_rank < cp_world")
    dev = kv_indices.device
    lens = seq_lens.to(torch.int64)
    ptr = kv_indptr.to(torch.int64)
    batch = lens.numel()
    cap = ptr[1:] - ptr[:-1]
    req = torch.repeat_interleave(torch.arange(batch, device=dev), cap)
    pos = torch.arange(ptr[-1].item() if batch else 0, device=dev) - ptr[:-1][req]
    keep = (pos < lens[req]) & (pos % cp_world == cp_rank)
    local_idx = kv_indices[: pos.numel()][keep].to(torch.int32).contiguous()
    local_lens = torch.zeros(batch, dtype=torch.int64, device=dev)
    local_lens.index_add_(0, req[keep], torch.ones_like(req[keep]))
    local_ptr = torch.zeros(batch + 1, dtype=torch.int64, device=dev)
    local_ptr[1:] = torch.cumsum(local_lens, 0)
    return (local_lens.to(torch.int32), local_idx, local_ptr.to(torch.int32),
            seq_lens.to(torch.int32).clone())


def all_gather_shares(o: torch.Tensor, lse: torch.Tensor,
                      group: Optional[dist.ProcessGroup] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """The exchange step: every rank receives every rank's share, rank-major,
    the layout ``mla_dcp_lse_merge_ranks`` reads: (parts [W, *o.shape],
    lses [W, *lse.shape])."""
    world = dist.get_world_size(group)
    parts = torch.empty((world,) + tuple(o.shape), dtype=o.dtype, device=o.device)
    lses = torch.empty((world,) + tuple(lse.shape), dtype=lse.dtype, device=lse.device)
    dist.all_gather(list(parts.unbind(0)), o.contiguous(), group=group)
    dist.all_gather(list(lses.unbind(0)), lse.contiguous(), group=group)
    return parts, lses


def dcp_decode_step(plan, q_lat, q_pe, pool, seq_lens, kv_indices, kv_indptr, glen,
                    scale: float, kv_scale: float, group: Optional[dist.ProcessGroup] = None,
                    workspace_t=None, share_dtype=torch.float32):
    """One DCP decode step on this rank: the rank's share (``mla_decode_dcp``),
    the all-gather of the shares, and their merge (``mla_dcp_lse_merge_ranks``),
    all on torch's current stream, which the collective orders itself against.
    Shares travel as fp32 by default, so the merged bf16 output is rounded once
    (bf16 shares halve the exchange and round twice).  The page table is the
    rank's own; returns the merged (o bf16, lse) for every row."""
    from . import mla
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    o, lse = mla.mla_decode_dcp(plan, q_lat, q_pe, pool, seq_lens, kv_indices, kv_indptr,
                                scale, kv_scale, glen, rank, world, workspace_t=workspace_t,
                                out_dtype=share_dtype if world > 1 else torch.bfloat16)
    if world == 1:
        return o, lse
    parts, lses = all_gather_shares(o, lse, group)
    return mla.mla_dcp_lse_merge_ranks(parts, lses)
