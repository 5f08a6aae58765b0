"""Python side of the double-precision oracle for paged gated-MLA decode.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Every function here is a
plain restatement of what the pages define; the heavy loop (scores, softmax and
the latent sum) lives in ``plmla_oracle.c`` and is reached through ctypes.

Passages followed:
  * Gated MLA is full softmax attention over cached compressed latent rows,
    with a gate on its output (TokenSpeed Kimi K3 post, architecture list).
  * The output gate is a sigmoid (TokenSpeed AgentX post, section "Kernel fusion
    and overlap complete the decode path", normalization/gating bullet).
  * Flat page pool of 1,536-token MLA pages addressed by one global page ID
    (TokenSpeed Kimi K3 post, section "A Generic, Unified Flat KV Layout for
    Cache Management").
  * Per-request KV splitting (TokenSpeed AgentX post, "Balance MLA work with
    per-request KV splitting", Figure 4).
  * Partial-softmax combine of split chunks (TokenSpeed Kimi K3 post, "Gated MLA"
    decode paragraph; decode context parallelism in the AgentX post, "AgentX
    benchmark results").
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle_plmla.so")
_lib = None

DC = 512          # latent width (BASELINE workload)
DR = 64           # rope width
PAGE_TOKENS = 1536  # tokens per MLA page (flat KV layout section)


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(
            os.path.join(_HERE, "plmla_oracle.c")):
        from .build import build_oracle
        build_oracle()
    lib = ctypes.CDLL(_LIB_PATH)
    i64, p = ctypes.c_int64, ctypes.c_void_p
    lib.oracle_attend_rows.restype = ctypes.c_int
    lib.oracle_attend_rows.argtypes = [p, p, p, i64, i64, i64, i64, p, i64, p, i64, i64, i64,
                                       i64, i64, ctypes.c_double, p, i64, i64, i64, p, p,
                                       ctypes.c_int]
    _lib = lib
    return lib


def _u16(a) -> np.ndarray:
    """bf16 data as a contiguous uint16 numpy array (accepts torch bf16 tensors)."""
    if hasattr(a, "view") and hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch
        a = a.detach().contiguous().cpu().view(torch.int16).numpy()
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        a = a.view(np.uint16)
    return a


def _i32(a) -> np.ndarray:
    if hasattr(a, "cpu"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def default_threads() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def attend_rows(q_nope, q_rope, slab, page_table, seq_lens, n_q, num_heads, scale, *,
                num_pages, page_stride=None, page_tokens=PAGE_TOKENS, dc=DC, dr=DR,
                rows=None, t_lo=0, t_hi=None, threads=None):
    """Ungated softmax attention over the paged latent history.

    Returns (o, lse): o is [n_rows, dc] float64, lse is [n_rows] float64
    (natural log; -inf where the row sees no token).  ``rows`` lists flat row
    ids (r*n_q + j)*H + h; None means every row in that order.  ``[t_lo, t_hi)``
    restricts the tokens (a KV chunk); the causal limit of draft token j is
    seq_lens[r] - (n_q - 1 - j).
    """
    lib = _load()
    qn, qr, sl = _u16(q_nope), _u16(q_rope), _u16(slab)
    pt, lens = _i32(page_table), _i32(seq_lens)
    R = lens.shape[0]
    if pt.ndim == 1:
        pt = pt.reshape(R, -1)
    table_ld = pt.shape[1] if pt.size else 1
    row_elems = dc + dr
    if page_stride is None:
        page_stride = page_tokens * row_elems
    if rows is None:
        n_rows = R * n_q * num_heads
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n_rows = rows_arr.shape[0]
    o = np.zeros((n_rows, dc), dtype=np.float64)
    lse = np.zeros((n_rows,), dtype=np.float64)
    if t_hi is None:
        t_hi = np.iinfo(np.int64).max
    rc = lib.oracle_attend_rows(
        qn.ctypes.data, qr.ctypes.data, sl.ctypes.data, num_pages, page_stride, page_tokens,
        row_elems, pt.ctypes.data, table_ld, lens.ctypes.data, R, n_q, num_heads, dc, dr,
        float(scale), rows_arr.ctypes.data if rows_arr is not None else None, n_rows,
        int(t_lo), int(t_hi), o.ctypes.data, lse.ctypes.data, int(threads or default_threads()))
    if rc == -1:
        raise IndexError("page table entry outside the pool")
    if rc != 0:
        raise MemoryError("oracle allocation failed")
    return o, lse


def gate_sigmoid(o, gate_logits):
    """out = sigmoid(g) * o elementwise, sigmoid(x) = 1 / (1 + e^-x), in double."""
    g = np.asarray(gate_logits, dtype=np.float64)
    return np.asarray(o, dtype=np.float64) / (1.0 + np.exp(-g))


def lse_merge(o_parts, lse_parts):
    """Merge partial softmax states of disjoint KV chunks.

    o_parts [S, n, dc] (each normalised by its own chunk), lse_parts [S, n].
    lse = ln sum_i e^{lse_i};  o = sum_i e^{lse_i - lse} o_i.  Rows where every
    chunk is empty (all lse_i = -inf) give o = 0 and lse = -inf.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    S, n = lse_parts.shape
    o = np.zeros(o_parts.shape[1:], dtype=np.float64)
    lse = np.full((n,), -np.inf)
    for row in range(n):
        m = max(lse_parts[:, row]) if S else -np.inf
        if m == -np.inf:
            continue
        w = [math.exp(lse_parts[i, row] - m) for i in range(S)]
        total = sum(w)
        lse[row] = m + math.log(total)
        for i in range(S):
            o[row] += (w[i] / total) * o_parts[i, row]
    return o, lse


def mla_decode_reference(q_nope, q_rope, gate, slab, page_table, seq_lens, n_q, num_heads,
                         scale, *, num_pages, page_stride=None, page_tokens=PAGE_TOKENS,
                         dc=DC, dr=DR, rows=None, threads=None):
    """Gated MLA decode: (out, lse) with out = sigmoid(gate) * softmax-attended latent.

    out is [n_rows, dc] float64 (before the final bf16 rounding), lse [n_rows]
    float64 taken before the gate.  ``gate`` holds [R*n_q, H, dc] logits.
    """
    o, lse = attend_rows(q_nope, q_rope, slab, page_table, seq_lens, n_q, num_heads, scale,
                         num_pages=num_pages, page_stride=page_stride,
                         page_tokens=page_tokens, dc=dc, dr=dr, rows=rows, threads=threads)
    g = _u16(gate).astype(np.uint32) << 16
    g = g.view(np.float32).astype(np.float64).reshape(-1, dc)
    if rows is not None:
        g = g[np.asarray(rows, dtype=np.int64)]
    return gate_sigmoid(o, g), lse


# --------------------------------------------------------------------------
# Split planning (TokenSpeed AgentX post, "Balance MLA work with per-request KV
# splitting", Figure 4): a target chunk length comes from the batch's total
# history and its parallelism budget; each request then gets as many chunks as
# its own history needs, so long histories get more splits.
# --------------------------------------------------------------------------

def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def plan_splits(seq_lens, budget: int, tile: int):
    """Return (chunk, splits) for the given per-request histories.

    chunk starts at ceil(sum L / budget) rounded up to the tile, and grows one
    tile at a time while the chunks do not fit the budget (sum_r ceil(L_r /
    chunk) > budget), stopping once every request is a single chunk.  A request
    with L = 0 gets no chunk.  Split s of request r covers tokens
    [s*chunk, min((s+1)*chunk, L_r)).
    """
    lens = [int(x) for x in seq_lens]
    if budget < 1 or tile < 1:
        raise ValueError("budget and tile must be positive")
    total = sum(lens)
    if total == 0:
        return tile, [0] * len(lens)
    chunk = _ceil_div(_ceil_div(total, budget), tile) * tile
    longest = _ceil_div(max(lens), tile) * tile

    def count(c):
        return sum(_ceil_div(L, c) for L in lens if L > 0)

    while count(chunk) > budget and chunk < longest:
        chunk += tile
    return chunk, [_ceil_div(L, chunk) if L > 0 else 0 for L in lens]


def split_budget(num_reqs: int, row_groups: int, cta_slots: int, min_splits: int,
                 chunks_per_member: int = 26, limit: int = 4096) -> int:
    """Chunk budget derived from the machine: 26 chunks for every persistent CTA
    of a row group (the finer the chunks, the closer each CTA's share of the
    work comes to its target), or enough for ``min_splits`` chunks per request
    if that is more, capped at ``limit``.  A hard-coded budget left most of a
    large GPU idle at batch 1 (AgentX - InferenceXv3 report, context-parallel
    section on in-GPU parallelism limits).  Raises ValueError when the
    per-request minimum alone is above ``limit``."""
    members = max(1, cta_slots // row_groups)
    wanted = num_reqs * max(1, min_splits)
    if wanted > limit:
        raise ValueError("budget above the planner's limit")
    budget = min(max(chunks_per_member * members, wanted), limit)
    return budget


# --------------------------------------------------------------------------
# KV append (vLLM blog "Kimi K3 Inference Backend Evolution", section "State
# Overwrite: How KDA Breaks Traditional KV Cache", the append-only contract of
# MLA: a new token's latent and rope rows are written after the request's
# existing history and no earlier row changes), into the flat page pool
# (TokenSpeed Kimi K3 post, "A Generic, Unified Flat KV Layout for Cache
# Management": one global page ID per 1,536-token page).
# --------------------------------------------------------------------------

def kv_append(slab, page_table, seq_lens, latent_new, rope_new, n_new, *,
              page_tokens=PAGE_TOKENS, page_stride=None, dc=DC, dr=DR):
    """Return a copy of the slab with each request's n_new new rows written.

    seq_lens counts the history after the append, so new token j of request r
    goes to position p = seq_lens[r] - n_new + j: page page_table[r, p //
    page_tokens], row p % page_tokens.  latent_new is [R*n_new, dc] and rope_new
    [R*n_new, dr] (bf16, row r*n_new + j); the stored row is latent then rope.
    Raises IndexError for a position below zero or a page ID outside the pool.
    """
    sl = _u16(slab).copy()
    shape = sl.shape
    flat = sl.reshape(-1)
    pt, lens = _i32(page_table), _i32(seq_lens)
    R = lens.shape[0]
    if pt.ndim == 1:
        pt = pt.reshape(R, -1)
    row_elems = dc + dr
    if page_stride is None:
        page_stride = page_tokens * row_elems
    num_pages = flat.size // page_stride
    lat = _u16(latent_new).reshape(R * n_new, dc)
    rope = _u16(rope_new).reshape(R * n_new, dr)
    for r in range(R):
        for j in range(n_new):
            p = int(lens[r]) - n_new + j
            if p < 0:
                raise IndexError("new token before the start of the history")
            page = int(pt[r, p // page_tokens])
            if page < 0 or page >= num_pages:
                raise IndexError("page table entry outside the pool")
            base = page * page_stride + (p % page_tokens) * row_elems
            flat[base:base + dc] = lat[r * n_new + j]
            flat[base + dc:base + row_elems] = rope[r * n_new + j]
    return flat.reshape(shape)
