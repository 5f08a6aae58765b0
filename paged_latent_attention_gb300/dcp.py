"""Decode context parallelism: one request's history split across GPUs.

Each of ``world`` ranks holds, for every request, a contiguous run of page-table
columns -- pages [rank * S, (rank + 1) * S) -- and decodes only those tokens with
mla_decode (its own plan, split decode and gated combine); one all-gather brings
every rank's gated output and log-sum-exp together and mla_merge_partials merges
them (TokenSpeed AgentX post, "AgentX benchmark results": decode context
parallelism, ranks combine partial attention results).  This shards the KV
pool's capacity and bandwidth for histories that one GPU cannot hold or stream
fast enough, at the price of one exchange of T x H x (512 bf16 + 1 fp32) per rank.

The split is by page-table columns, identical for every request, so a rank's
share is a plain strided view of the table and a clamp of the lengths, computed
on the device (no host round trip per step).  Only single-token decode is
sharded: with draft tokens the causal limit falls in the last rank's part only,
which the per-rank decode cannot tell from a history that ends there.
"""
from __future__ import annotations

import math

import torch

from . import api

PAGE_TOKENS = api.PAGE_TOKENS


def pages_per_rank(table_cols: int, world: int) -> int:
    """Page-table columns each rank owns (the last rank may own fewer)."""
    if world < 1 or table_cols < 1:
        raise ValueError("world and table columns must be positive")
    return math.ceil(table_cols / world)


def shard_bounds(rank: int, world: int, table_cols: int, page_tokens: int = PAGE_TOKENS):
    """Token range [t_lo, t_hi) of every request that rank `rank` decodes."""
    if not 0 <= rank < world:
        raise ValueError("rank outside the group")
    s = pages_per_rank(table_cols, world)
    return rank * s * page_tokens, (rank + 1) * s * page_tokens


def shard_view(page_table, seq_lens, rank: int, world: int, page_tokens: int = PAGE_TOKENS):
    """Rank `rank`'s page table (a column view of the full one, same row stride)
    and history lengths (device tensors, no synchronisation)."""
    cols = page_table.shape[1]
    s = pages_per_rank(cols, world)
    first = rank * s
    # a rank past the last column sees no tokens; any valid column start serves
    table_k = page_table[:, min(first, cols - 1):]
    t_lo, t_hi = shard_bounds(rank, world, cols, page_tokens)
    lens_k = (seq_lens.to(torch.int64) - t_lo).clamp_(0, t_hi - t_lo).to(torch.int32)
    return table_k, lens_k


def decode_shard(q_nope_absorbed, q_rope, gate, slab, page_table, seq_lens, rank, world, *,
                 kv_scale=None, scale=api.DEFAULT_SCALE, workspace=None, stream=None):
    """Rank `rank`'s gated part (out_k, lse_k): mla_decode (mla_decode_fp8 when
    `kv_scale` is given and the slab holds E4M3 codes) on its column view."""
    table_k, lens_k = shard_view(page_table, seq_lens, rank, world)
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
