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

DC = 512          # compressed latent width of the MLA cache rows
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
    dbl, c_int = ctypes.c_double, ctypes.c_int
    lib.oracle_attend_rows.restype = c_int
    lib.oracle_attend_rows.argtypes = [p, p, p, c_int, dbl, i64, i64, i64, i64, p, i64, p, i64,
                                       i64, i64, i64, i64, dbl, p, i64, i64, i64, p, p, p, p, p,
                                       p, p, c_int]
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


def _u8(a) -> np.ndarray:
    """Byte data (E4M3 codes) as a contiguous uint8 numpy array (accepts torch
    uint8 / float8 tensors)."""
    if hasattr(a, "detach"):
        import torch
        a = a.detach().contiguous().cpu()
        if a.dtype != torch.uint8:
            a = a.view(torch.uint8)
        a = a.numpy()
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8:
        a = a.view(np.uint8)
    return a


def _as_f64(a) -> np.ndarray:
    """Query values as contiguous float64: bf16 (torch tensor or uint16 bit
    patterns) widened exactly, any float array converted."""
    if hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        return np.ascontiguousarray(_bf16_to_f64(a))
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return np.ascontiguousarray(_bf16_to_f64(a))
    return np.ascontiguousarray(a, dtype=np.float64)


def _rows_f64(q, rows, width) -> np.ndarray:
    """[total rows, width] float64 holding the listed rows of q (the rest zero)."""
    if hasattr(q, "detach"):
        import torch
        flat = q.detach().reshape(-1, width)
        total = flat.shape[0]
        idx = torch.as_tensor(rows, dtype=torch.long, device=flat.device)
        picked = _as_f64(flat.index_select(0, idx).contiguous())
    else:
        flat = np.asarray(q).reshape(-1, width)
        total = flat.shape[0]
        picked = _as_f64(np.ascontiguousarray(flat[rows]))
    out = np.zeros((total, width), dtype=np.float64)
    out[rows] = picked
    return out


def _i32(a) -> np.ndarray:
    if hasattr(a, "cpu"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def default_threads() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def _bf16_to_f64(a) -> np.ndarray:
    """bf16 bit patterns (or a torch bf16 tensor) widened exactly to float64."""
    u = _u16(a).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def attend_rows(q_nope, q_rope, slab, page_table, seq_lens, n_q, num_heads, scale, *,
                num_pages, page_stride=None, page_tokens=PAGE_TOKENS, dc=DC, dr=DR,
                rows=None, t_lo=0, t_hi=None, threads=None, kv_format="bf16", kv_scale=1.0,
                with_abs=False, query_err=None):
    """Ungated softmax attention over the paged latent history.

    Returns (o, lse), or (o, lse, extra) with ``with_abs``: o is [n_rows, dc]
    float64, lse is [n_rows] float64 (natural log; -inf where the row sees no
    token); extra is a dict of sensitivity terms: "o_abs" = sum_t w_t |c_t|
    (the probability-weighted absolute latent, [n_rows, dc]), "abs_sum" =
    sum_t |c_t| ([n_rows, dc]), "w_max" = the largest weight ([n_rows]) and,
    given ``query_err`` ([R*n_q*H, dc + dr] bounds on the error of each query
    element), "d_max" = max_t |scale| sum_d query_err[d] |x_t[d]|, the largest
    bound on a score's error ([n_rows]).
    ``rows`` lists flat row ids (r*n_q + j)*H + h; None means every row in that
    order.  ``[t_lo, t_hi)`` restricts the tokens (a KV chunk); the causal limit
    of draft token j is seq_lens[r] - (n_q - 1 - j).  The queries are bf16 (or
    any float array, taken as float64).  ``kv_format`` "e4m3": the slab holds
    E4M3 bytes and an element's value is kv_scale times the decoded byte.
    """
    lib = _load()
    if rows is None:
        qn, qr = _as_f64(q_nope), _as_f64(q_rope)
    else:
        # only the requested rows are widened; the others are never read
        sel = np.asarray(rows, dtype=np.int64)
        qn, qr = _rows_f64(q_nope, sel, dc), _rows_f64(q_rope, sel, dr)
    if kv_format == "bf16":
        sl, fp8 = _u16(slab), 0
    elif kv_format == "e4m3":
        sl, fp8 = _u8(slab), 1
    else:
        raise ValueError(kv_format)
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
    extra = None
    eps = None
    if with_abs:
        extra = {"o_abs": np.zeros((n_rows, dc)), "abs_sum": np.zeros((n_rows, dc)),
                 "w_max": np.zeros((n_rows,)), "d_max": np.zeros((n_rows,))}
        if query_err is not None:
            eps = np.ascontiguousarray(np.asarray(query_err, dtype=np.float64)
                                       .reshape(R * n_q * num_heads, row_elems))
    if t_hi is None:
        t_hi = np.iinfo(np.int64).max

    def ptr(a):
        return a.ctypes.data if a is not None else None
    rc = lib.oracle_attend_rows(
        qn.ctypes.data, qr.ctypes.data, sl.ctypes.data, fp8, float(kv_scale), num_pages,
        page_stride, page_tokens, row_elems, pt.ctypes.data, table_ld, lens.ctypes.data, R, n_q,
        num_heads, dc, dr, float(scale), ptr(rows_arr), n_rows, int(t_lo), int(t_hi),
        o.ctypes.data, ptr(extra["o_abs"]) if extra else None, lse.ctypes.data, ptr(eps),
        ptr(extra["abs_sum"]) if extra else None, ptr(extra["w_max"]) if extra else None,
        ptr(extra["d_max"]) if extra else None, int(threads or default_threads()))
    if rc == -1:
        raise IndexError("page table entry outside the pool")
    if rc != 0:
        raise MemoryError("oracle allocation failed")
    return (o, lse, extra) if with_abs else (o, lse)


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


def plan_splits_uniform(seq_lens, budget: int, tile: int):
    """The uniform baseline of the same section (Figure 4, left panel; the
    comparison of Figure 5): every request with history gets the same number of
    chunks, su = budget // (requests with history), at least 1.  Returns
    (chunks, splits): request r's chunk ceil(L_r / su) rounded up to the tile,
    and its split count ceil(L_r / chunk_r) (0 and 0 for L_r = 0)."""
    lens = [int(x) for x in seq_lens]
    if budget < 1 or tile < 1:
        raise ValueError("budget and tile must be positive")
    live = sum(1 for L in lens if L > 0)
    su = max(1, budget // max(1, live))
    chunks, splits = [], []
    for L in lens:
        if L == 0:
            chunks.append(0)
            splits.append(0)
            continue
        c = _ceil_div(_ceil_div(L, su), tile) * tile
        chunks.append(c)
        splits.append(_ceil_div(L, c))
    return chunks, splits


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


# --------------------------------------------------------------------------
# FP8 pages.  The deployment keeps its MLA cache in FP8 (TokenSpeed AgentX post,
# memory-budget paragraph: FP8 target/drafter KV cache), and the AMD notes of
# the AgentX - InferenceXv3 report name the encoding (float8_e4m3fn, as opposed
# to gfx942's e4m3fnuz).  The pages give no scale granularity; the reading here
# is one float scale per cache tensor: element value = kv_scale * decoded byte.
# The pages say nothing about the query: the definition keeps it bf16, so the
# reference below is attention of the bf16 query over the dequantised cache.
# quantize_query_rows restates the library's own query split (a documented
# library function with no counterpart on the pages) only to check that
# function bit for bit.
# --------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """E4M3 bytes -> float64: sign bit, 4 exponent bits (bias 7), 3 mantissa
    bits; exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN."""
    c = _u8(codes).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    v = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    v = np.where((e == 15) & ((c & 7) == 7), np.nan, v)
    return sign * v


_E4M3_POS = None


def _e4m3_table() -> np.ndarray:
    global _E4M3_POS
    if _E4M3_POS is None:
        _E4M3_POS = e4m3_decode(np.arange(127, dtype=np.uint8))   # 0 .. 448, increasing
    return _E4M3_POS


def e4m3_encode(x) -> np.ndarray:
    """Round float values to E4M3 bytes: nearest representable magnitude, ties
    to the even code, magnitudes above 448 saturated to 448, NaN -> 0x7F, the
    sign kept (also for a zero result)."""
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    tab = _e4m3_table()
    hi = np.clip(np.searchsorted(tab, np.minimum(ax, E4M3_MAX), side="left"), 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    d_lo = np.minimum(ax, E4M3_MAX) - tab[lo]
    d_hi = tab[hi] - np.minimum(ax, E4M3_MAX)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def query_scale_exponent(amax) -> np.ndarray:
    """Per-row power-of-two scale 2^e of the FP8 query: the smallest e with
    amax * 2^-e <= 448 (E4M3's largest finite value), e >= -126; e = 0 for an
    all-zero row."""
    amax = np.asarray(amax, dtype=np.float64)
    f, E = np.frexp(amax)                    # amax = f * 2^E, f in [0.5, 1)
    k = E - 1                                # amax = (2f) * 2^k, 2f in [1, 2)
    e = np.where(2.0 * f <= 1.75, k - 8, k - 7)
    e = np.maximum(e, -126)
    return np.where(amax == 0, 0, e).astype(np.int32)


def quantize_query_rows(q_nope, q_rope):
    """The library's two-part FP8 query (checker of mla_quantize_queries_fp8):
    each row of [q_nope | q_rope] (dc + dr values) is scaled by 2^-e, e =
    query_scale_exponent(max |q| over the row); hi = E4M3 code of v = q * 2^-e,
    lo = E4M3 code of v - decode(hi) (both round to nearest even).  Returns
    (hi [rows, dc + dr] uint8, lo [rows, dc + dr] uint8, exps [rows] int32)."""
    qn, qr = _as_f64(q_nope), _as_f64(q_rope)
    qn = qn.reshape(-1, qn.shape[-1])
    qr = qr.reshape(-1, qr.shape[-1])
    q = np.concatenate([qn, qr], axis=1)
    e = query_scale_exponent(np.max(np.abs(q), axis=1))
    v = np.ldexp(q, -e[:, None].astype(np.int64))
    hi = e4m3_encode(v)
    lo = e4m3_encode(v - e4m3_decode(hi))
    return hi, lo, e


def dequantize_query_rows(hi, lo, exps) -> np.ndarray:
    """float64 values of two-part FP8 query rows: (decode(hi) + decode(lo)) * 2^e."""
    return np.ldexp(e4m3_decode(hi) + e4m3_decode(lo),
                    np.asarray(exps, dtype=np.int64)[:, None])


def mla_decode_e4m3_reference(q_nope, q_rope, gate, slab8, kv_scale, page_table, seq_lens, n_q,
                              num_heads, scale, *, num_pages, page_stride=None,
                              page_tokens=PAGE_TOKENS, dc=DC, dr=DR, rows=None, threads=None,
                              with_abs=False, query_err=None):
    """Gated MLA decode over E4M3 pages: the bf16 query, exactly, attending over
    the dequantised cache (kv_scale * decoded byte), then the sigmoid gate.

    Returns (out, lse), or with ``with_abs`` (out, lse, terms) where terms holds
    the gated sensitivity terms "A" = sigmoid(g) * sum_t w_t |c_t|, "B" =
    sigmoid(g) * w_max * sum_t |c_t| and "D" (per row, the bound on a score's
    error for the per-element query errors ``query_err``, 0 without it); see
    attend_rows."""
    res = attend_rows(q_nope, q_rope, slab8, page_table, seq_lens, n_q, num_heads, scale,
                      num_pages=num_pages, page_stride=page_stride, page_tokens=page_tokens,
                      dc=dc, dr=dr, rows=rows, threads=threads, kv_format="e4m3",
                      kv_scale=kv_scale, with_abs=with_abs, query_err=query_err)
    g = _bf16_to_f64(gate).reshape(-1, dc)
    if rows is not None:
        g = g[np.asarray(rows, dtype=np.int64)]
    out = gate_sigmoid(res[0], g)
    if not with_abs:
        return out, res[1]
    x = res[2]
    terms = {"A": gate_sigmoid(x["o_abs"], g),
             "B": gate_sigmoid(x["w_max"][:, None] * x["abs_sum"], g),
             "D": x["d_max"]}
    return out, res[1], terms


def kv_append_e4m3(slab8, page_table, seq_lens, latent_new, rope_new, n_new, kv_scale, *,
                   page_tokens=PAGE_TOKENS, page_stride=None, dc=DC, dr=DR):
    """kv_append into E4M3 pages: each new bf16 value x is stored as the E4M3
    code of x / kv_scale, the quotient taken in float32 (x and kv_scale as
    float32, one correctly rounded division).  Positions, pages and errors as in
    kv_append."""
    sl = _u8(slab8).copy()
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
    s32 = np.float32(kv_scale)
    lat = (_bf16_to_f64(latent_new).astype(np.float32) / s32).reshape(R * n_new, dc)
    rope = (_bf16_to_f64(rope_new).astype(np.float32) / s32).reshape(R * n_new, dr)
    lat_c, rope_c = e4m3_encode(lat), e4m3_encode(rope)
    for r in range(R):
        for j in range(n_new):
            p = int(lens[r]) - n_new + j
            if p < 0:
                raise IndexError("new token before the start of the history")
            page = int(pt[r, p // page_tokens])
            if page < 0 or page >= num_pages:
                raise IndexError("page table entry outside the pool")
            base = page * page_stride + (p % page_tokens) * row_elems
            flat[base:base + dc] = lat_c[r * n_new + j]
            flat[base + dc:base + row_elems] = rope_c[r * n_new + j]
    return flat.reshape(shape)
