"""Decode context parallelism: one request's history split across GPUs.

Each of ``world`` ranks holds, for every request, every world-th page of its
history -- page column c of request r belongs to rank (c + r) mod world -- and
decodes only those tokens with mla_decode (its own plan, split decode and gated
combine); one all-gather brings every rank's gated output and log-sum-exp
together and mla_merge_partials merges them (TokenSpeed AgentX post, "AgentX
benchmark results": decode context parallelism, ranks combine partial attention
results).  This shards the KV pool's capacity and bandwidth for histories that
one GPU cannot hold or stream fast enough, at the price of one exchange of
T x H x (512 bf16 + 1 fp32) per rank.

Dealing pages round-robin gives every rank the same number of a request's pages
up to one, and rotating the first rank with the request spreads the leftover
pages over the ranks, so the ranks stream nearly the same number of tokens
(the softmax does not depend on the order of the tokens, so a rank's pages
form one local history).  A rank's table rows and lengths are built on the
device by mla_dcp_shard (no host round trip per step).  Only single-token
decode is sharded: with draft tokens the causal limit falls on the request's
last tokens, which one rank alone holds.
"""
from __future__ import annotations

import torch

from . import api

PAGE_TOKENS = api.PAGE_TOKENS


def owner(column: int, request: int, world: int) -> int:
    """The rank that holds page column `column` of request `request`."""
    return (column + request) % world


def shard_view(page_table, seq_lens, rank: int, world: int, stream=None):
    """Rank `rank`'s page table ([R, ceil(ld / world)], its pages in column
    order) and history lengths (device tensors, no synchronisation)."""
    if not 0 <= rank < world:
        raise ValueError("rank outside the group")
    return api.mla_dcp_shard(page_table, seq_lens, world, rank, stream=stream)


def decode_shard(q_nope_absorbed, q_rope, gate, slab, page_table, seq_lens, rank, world, *,
                 kv_scale=None, scale=api.DEFAULT_SCALE, workspace=None, stream=None):
    """Rank `rank`'s gated part (out_k, lse_k): mla_decode (mla_decode_fp8 when
    `kv_scale` is given and the slab holds E4M3 codes) on its pages."""
    table_k, lens_k = shard_view(page_table, seq_lens, rank, world, stream=stream)
    if kv_scale is None:
        return api.mla_decode(q_nope_absorbed, q_rope, gate, slab, table_k, lens_k, n_q=1,
                              scale=scale, workspace=workspace, stream=stream)
    return api.mla_decode_fp8(q_nope_absorbed, q_rope, gate, slab, table_k, lens_k,
                              kv_scale=kv_scale, n_q=1, scale=scale, workspace=workspace,
                              stream=stream)


def dcp_decode(q_nope_absorbed, q_rope, gate, slab, page_table, seq_lens, *, group=None,
               kv_scale=None, scale=api.DEFAULT_SCALE, workspace=None, stream=None):
    """mla_decode of single-token requests with every history split across the
    ranks of `group` (torch.distributed); every rank returns the full (out, lse).
    With `kv_scale`, the slab holds E4M3 pages (the merge is the same: each part
    is a gated output with its LSE, whatever the page format)."""
    import torch.distributed as dist

    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    out_k, lse_k = decode_shard(q_nope_absorbed, q_rope, gate, slab, page_table, seq_lens, rank,
                                world, kv_scale=kv_scale, scale=scale, workspace=workspace,
                                stream=stream)
    out_parts = torch.empty((world,) + tuple(out_k.shape), dtype=out_k.dtype, device=out_k.device)
    lse_parts = torch.empty((world,) + tuple(lse_k.shape), dtype=lse_k.dtype, device=lse_k.device)
    dist.all_gather_into_tensor(out_parts, out_k, group=group)
    dist.all_gather_into_tensor(lse_parts, lse_k, group=group)
    return api.mla_merge_partials(out_parts, lse_parts, stream=stream)
