"""Torch-tensor front end of libplmla (argument marshalling only).

Every step of the decode runs in the CUDA library; these functions check
shapes, dtypes and devices, then pass raw device pointers and sizes through the
C ABI.  PyTorch only supplies device memory and the current stream.
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _native

LATENT = 512
ROPE = 64
ROW = LATENT + ROPE
PAGE_TOKENS = 1536
DEFAULT_SCALE = 1.0 / math.sqrt(192.0)   # a 128-wide nope + 64-wide rope head


def _stream_ptr(stream, device):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes_void(s.cuda_stream)


def ctypes_void(v):
    return None if v in (0, None) else int(v)


def _require(cond, msg):
    if not cond:
        raise ValueError(msg)


def _check_bf16(t, name, shape=None):
    _require(isinstance(t, torch.Tensor), f"{name} must be a tensor")
    _require(t.is_cuda, f"{name} must be a CUDA tensor")
    _require(t.dtype == torch.bfloat16, f"{name} must be bfloat16")
    _require(t.is_contiguous(), f"{name} must be contiguous")
    if shape is not None:
        _require(tuple(t.shape) == tuple(shape), f"{name} has shape {tuple(t.shape)}, "
                                                 f"expected {tuple(shape)}")


def mla_split_budget(num_reqs, n_q, num_heads, cta_budget=0, min_splits=1) -> int:
    b = _native.lib().mla_split_budget(num_reqs, n_q, num_heads, cta_budget, min_splits)
    if b < 1:
        raise ValueError("invalid shape for mla_split_budget")
    return int(b)


def mla_workspace_size(num_reqs, n_q, num_heads, cta_budget=0, min_splits=1) -> int:
    n = _native.lib().mla_workspace_size(num_reqs, n_q, num_heads, cta_budget, min_splits)
    if n == 0:
        raise ValueError("invalid shape for mla_workspace_size")
    return int(n)


def mla_workspace_size_fp8(num_reqs, n_q, num_heads, cta_budget=0, min_splits=1) -> int:
    n = _native.lib().mla_workspace_size_fp8(num_reqs, n_q, num_heads, cta_budget, min_splits)
    if n == 0:
        raise ValueError("invalid shape for mla_workspace_size_fp8")
    return int(n)


def allocate_workspace(num_reqs, n_q, num_heads, cta_budget=0, min_splits=1, device=None,
                       fp8=False):
    """A caller-owned workspace tensor (uint8) of the size mla_decode (or, with
    ``fp8``, mla_decode_fp8) needs."""
    size = mla_workspace_size_fp8 if fp8 else mla_workspace_size
    n = size(num_reqs, n_q, num_heads, cta_budget, min_splits)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def _byte_view(slab):
    """An E4M3 slab as uint8 (float8_e4m3fn tensors are viewed, not copied)."""
    if slab.dtype == torch.uint8:
        return slab
    _require(slab.dtype == getattr(torch, "float8_e4m3fn", None),
             "an FP8 slab must be uint8 or float8_e4m3fn")
    return slab.view(torch.uint8)


def mla_decode(q_nope_absorbed, q_rope, gate, slab, page_table, seq_lens, *, n_q=1,
               scale=DEFAULT_SCALE, out=None, lse=None, workspace=None, cta_budget=0,
               min_splits=1, stream=None, with_lse=True, events=None):
    """One gated-MLA decode step; returns (out, lse).

    ``events`` (optional): four torch.cuda.Event (or None) recorded before the
    plan kernel, before the split-decode kernel, before the combine kernel and
    after it, on the launch stream.  Each event must have been recorded once
    already, so that torch has created its handle.

    q_nope_absorbed, gate: [R*n_q, H, 512] bf16; q_rope: [R*n_q, H, 64] bf16.
    slab: [num_pages, page_stride] bf16 (page_stride >= 1536*576; row r of a
    page at r*576).  page_table: [R, ld] int32 with unit column stride (its row
    stride is passed through, so a strided view works).  seq_lens: [R] int32.
    """
    return _decode(q_nope_absorbed, q_rope, gate, slab, page_table, seq_lens, None, n_q, scale,
                   out, lse, workspace, cta_budget, min_splits, stream, with_lse, events)


def mla_decode_fp8(q_nope_absorbed, q_rope, gate, slab, page_table, seq_lens, *, kv_scale,
                   n_q=1, scale=DEFAULT_SCALE, out=None, lse=None, workspace=None, cta_budget=0,
                   min_splits=1, stream=None, with_lse=True, events=None):
    """mla_decode over E4M3 pages: slab is [num_pages, page_stride] uint8 (or
    float8_e4m3fn) holding E4M3 codes of value / kv_scale, 576 bytes per token
    row (page_stride >= 1536*576, a multiple of 16).  The queries stay bf16;
    the library splits each query row into two E4M3 parts with a power-of-two
    scale (exact for elements above 2^-2 of the scale).
    The workspace must come from allocate_workspace(..., fp8=True)."""
    _require(math.isfinite(kv_scale) and kv_scale > 0, "kv_scale must be finite and > 0")
    return _decode(q_nope_absorbed, q_rope, gate, _byte_view(slab), page_table, seq_lens,
                   float(kv_scale), n_q, scale, out, lse, workspace, cta_budget, min_splits,
                   stream, with_lse, events)


def _decode(q_nope_absorbed, q_rope, gate, slab, page_table, seq_lens, kv_scale, n_q, scale,
            out, lse, workspace, cta_budget, min_splits, stream, with_lse, events):
    fp8 = kv_scale is not None
    _require(q_nope_absorbed.dim() == 3, "q_nope_absorbed must be [R*n_q, H, 512]")
    T, H, _ = q_nope_absorbed.shape
    _require(T % n_q == 0, "first dimension must be num_reqs * n_q")
    R = T // n_q
    device = q_nope_absorbed.device
    _check_bf16(q_nope_absorbed, "q_nope_absorbed", (T, H, LATENT))
    _check_bf16(q_rope, "q_rope", (T, H, ROPE))
    _check_bf16(gate, "gate", (T, H, LATENT))
    want = torch.uint8 if fp8 else torch.bfloat16
    _require(slab.is_cuda and slab.dtype == want and slab.dim() == 2,
             f"slab must be a 2-D CUDA {want} tensor [num_pages, page_stride]")
    _require(slab.stride(1) == 1, "slab pages must be contiguous")
    num_pages, page_stride = slab.shape[0], slab.stride(0)
    _require(slab.shape[1] >= PAGE_TOKENS * ROW, "slab page too small")
    _require(page_table.is_cuda and page_table.dtype == torch.int32 and page_table.dim() == 2,
             "page_table must be a 2-D CUDA int32 tensor")
    _require(page_table.shape[0] == R and page_table.stride(1) == 1,
             "page_table must be [R, ld] with unit column stride")
    _require(seq_lens.is_cuda and seq_lens.dtype == torch.int32 and seq_lens.is_contiguous()
             and tuple(seq_lens.shape) == (R,), "seq_lens must be a contiguous CUDA int32 [R]")
    if out is None:
        out = torch.empty_like(q_nope_absorbed)
    _check_bf16(out, "out", (T, H, LATENT))
    if lse is None and with_lse:
        lse = torch.empty(T, H, dtype=torch.float32, device=device)
    if lse is not None:
        _require(lse.is_cuda and lse.dtype == torch.float32 and lse.is_contiguous()
                 and tuple(lse.shape) == (T, H), "lse must be a contiguous CUDA fp32 [T, H]")
    if workspace is None:
        workspace = allocate_workspace(R, n_q, H, cta_budget, min_splits, device, fp8=fp8)
    _require(workspace.is_cuda and workspace.is_contiguous(), "workspace must be CUDA memory")
    nbytes = workspace.numel() * workspace.element_size()
    ev = None
    if events is not None:
        handles = []
        for e in events:
            h = None if e is None else int(e.cuda_event)
            _require(h != 0, "stage events must have been recorded once before use")
            handles.append(h)
        ev = _native.StageEvents(*handles)
    lib = _native.lib()
    head = (q_nope_absorbed.data_ptr(), q_rope.data_ptr(), gate.data_ptr(), slab.data_ptr(),
            num_pages, page_stride)
    tail = (page_table.data_ptr(), page_table.stride(0), seq_lens.data_ptr(), R, n_q, H,
            float(scale), out.data_ptr(), lse.data_ptr() if lse is not None else None,
            workspace.data_ptr(), nbytes, int(cta_budget), int(min_splits),
            _stream_ptr(stream, device), ctypes.byref(ev) if ev is not None else None)
    if fp8:
        status = lib.mla_decode_fp8_ex(*head, kv_scale, *tail)
    else:
        status = lib.mla_decode_ex(*head, *tail)
    _native.check(status, "mla_decode_fp8" if fp8 else "mla_decode")
    return out, lse


def mla_decode_layers(q_nope_absorbed, q_rope, gate, slabs, page_table, seq_lens, *, n_q=1,
                      scale=DEFAULT_SCALE, kv_scale=None, out=None, lse=None, workspace=None,
                      cta_budget=0, min_splits=1, stream=None, with_lse=True):
    """The decode step of several MLA layers that share the page table and the
    history lengths (every layer's pool is paged by the same global page IDs):
    one split plan for the step, then each layer's split decode and combine.
    q_nope_absorbed, q_rope, gate and slabs are lists with one tensor per layer,
    each as in mla_decode (E4M3 slabs with `kv_scale`, a float or one per
    layer); returns (outs, lses), lists (lses of None without LSE).  Layer l's
    results equal mla_decode's (or mla_decode_fp8's) on layer l's tensors."""
    L = len(slabs)
    _require(L >= 1 and len(q_nope_absorbed) == L and len(q_rope) == L and len(gate) == L,
             "one query, rope, gate and slab tensor per layer")
    fp8 = kv_scale is not None
    scales = None
    if fp8:
        scales = list(kv_scale) if isinstance(kv_scale, (list, tuple)) else [kv_scale] * L
        _require(len(scales) == L and all(math.isfinite(v) and v > 0 for v in scales),
                 "kv_scale must be finite and > 0 (one value, or one per layer)")
        slabs = [_byte_view(s) for s in slabs]
    qn0 = q_nope_absorbed[0]
    _require(qn0.dim() == 3, "q_nope_absorbed must be [R*n_q, H, 512]")
    T, H, _ = qn0.shape
    _require(T % n_q == 0, "first dimension must be num_reqs * n_q")
    R = T // n_q
    device = qn0.device
    want = torch.uint8 if fp8 else torch.bfloat16
    num_pages, page_stride = slabs[0].shape[0], slabs[0].stride(0)
    for l in range(L):
        _check_bf16(q_nope_absorbed[l], "q_nope_absorbed", (T, H, LATENT))
        _check_bf16(q_rope[l], "q_rope", (T, H, ROPE))
        _check_bf16(gate[l], "gate", (T, H, LATENT))
        s = slabs[l]
        _require(s.is_cuda and s.dtype == want and s.dim() == 2 and s.stride(1) == 1,
                 f"each slab must be a 2-D CUDA {want} tensor with contiguous pages")
        _require(s.shape[0] == num_pages and s.stride(0) == page_stride,
                 "the layers' slabs must share the page count and page stride")
    _require(slabs[0].shape[1] >= PAGE_TOKENS * ROW, "slab page too small")
    _require(page_table.is_cuda and page_table.dtype == torch.int32 and page_table.dim() == 2,
             "page_table must be a 2-D CUDA int32 tensor")
    _require(page_table.shape[0] == R and page_table.stride(1) == 1,
             "page_table must be [R, ld] with unit column stride")
    _require(seq_lens.is_cuda and seq_lens.dtype == torch.int32 and seq_lens.is_contiguous()
             and tuple(seq_lens.shape) == (R,), "seq_lens must be a contiguous CUDA int32 [R]")
    if out is None:
        out = [torch.empty_like(q) for q in q_nope_absorbed]
    _require(len(out) == L, "one output tensor per layer")
    for o in out:
        _check_bf16(o, "out", (T, H, LATENT))
    if lse is None and with_lse:
        lse = [torch.empty(T, H, dtype=torch.float32, device=device) for _ in range(L)]
    if lse is not None:
        _require(len(lse) == L, "one lse tensor per layer")
        for v in lse:
            _require(v is None or (v.is_cuda and v.dtype == torch.float32 and v.is_contiguous()
                                   and tuple(v.shape) == (T, H)),
                     "lse must be a contiguous CUDA fp32 [T, H] (or None)")
    if workspace is None:
        workspace = allocate_workspace(R, n_q, H, cta_budget, min_splits, device, fp8=fp8)
    _require(workspace.is_cuda and workspace.is_contiguous(), "workspace must be CUDA memory")
    nbytes = workspace.numel() * workspace.element_size()

    def ptrs(ts):
        arr = (ctypes.c_void_p * L)(*[None if t is None else t.data_ptr() for t in ts])
        return arr, ctypes.cast(arr, ctypes.c_void_p)

    keep = [ptrs(q_nope_absorbed), ptrs(q_rope), ptrs(gate), ptrs(slabs), ptrs(out)]
    lse_arr = ptrs(lse) if lse is not None else (None, None)
    lib = _native.lib()
    head = [L] + [k[1] for k in keep[:4]]
    tail = [num_pages, page_stride, page_table.data_ptr(), page_table.stride(0),
            seq_lens.data_ptr(), R, n_q, H, float(scale), keep[4][1], lse_arr[1],
            workspace.data_ptr(), nbytes, int(cta_budget), int(min_splits),
            _stream_ptr(stream, device)]
    if fp8:
        sc = (ctypes.c_float * L)(*[float(v) for v in scales])
        status = lib.mla_decode_layers_fp8(*head, ctypes.cast(sc, ctypes.c_void_p), *tail)
    else:
        status = lib.mla_decode_layers(*head, *tail)
    _native.check(status, "mla_decode_layers_fp8" if fp8 else "mla_decode_layers")
    return out, (lse if lse is not None else [None] * L)


def mla_quantize_queries_fp8(q_nope_absorbed, q_rope, stream=None):
    """The FP8 decode's query step: (hi [rows, 576] uint8, lo [rows, 576] uint8,
    exps [rows] int32) for the rows of [q_nope | q_rope] (any leading shape,
    flattened): q = (decode(hi) + decode(lo)) * 2^exp, exactly where
    |q| >= 2^(exp - 2)."""
    _require(q_nope_absorbed.is_cuda and q_nope_absorbed.dtype == torch.bfloat16
             and q_nope_absorbed.is_contiguous() and q_nope_absorbed.shape[-1] == LATENT,
             "q_nope_absorbed must be contiguous CUDA bf16 [..., 512]")
    rows = q_nope_absorbed.numel() // LATENT
    _require(q_rope.is_cuda and q_rope.dtype == torch.bfloat16 and q_rope.is_contiguous()
             and q_rope.numel() == rows * ROPE, "q_rope must be contiguous CUDA bf16 [..., 64]")
    codes = torch.empty(2, rows, ROW, dtype=torch.uint8, device=q_nope_absorbed.device)
    exps = torch.empty(rows, dtype=torch.int32, device=q_nope_absorbed.device)
    status = _native.lib().mla_quantize_queries_fp8(
        q_nope_absorbed.data_ptr(), q_rope.data_ptr(), rows, codes.data_ptr(), exps.data_ptr(),
        _stream_ptr(stream, q_nope_absorbed.device))
    _native.check(status, "mla_quantize_queries_fp8")
    return codes[0], codes[1], exps


def set_page_checks(on: bool) -> None:
    """Process-wide: check every page-table entry a decode step uses after the
    step (status 40 in the workspace's status word if one is out of range)."""
    _native.lib().mla_set_page_checks(1 if on else 0)


def get_page_checks() -> bool:
    return bool(_native.lib().mla_get_page_checks())


SPLIT_MODES = {"per-request": 0, "uniform": 1}


def set_split_mode(mode: str) -> None:
    """Process-wide split rule of the planner: "per-request" (the default) or
    "uniform" (the same split count for every request, the baseline of the
    pages' Figure 5 comparison)."""
    _require(mode in SPLIT_MODES, f"split mode must be one of {sorted(SPLIT_MODES)}")
    _native.check(_native.lib().mla_set_split_mode(SPLIT_MODES[mode]), "mla_set_split_mode")


def get_split_mode() -> str:
    m = int(_native.lib().mla_get_split_mode())
    return {v: k for k, v in SPLIT_MODES.items()}[m]


def set_team_clusters(max_teams: int) -> None:
    """Process-wide widest cluster (1, 2 or 4; default 2) of 64-row query teams
    that share each KV tile's load (TMA multicast) in the bf16 decode; the
    outputs do not depend on it."""
    _require(max_teams in (1, 2, 4), "max_teams must be 1, 2 or 4")
    _native.check(_native.lib().mla_set_team_clusters(int(max_teams)), "mla_set_team_clusters")


def get_team_clusters() -> int:
    return int(_native.lib().mla_get_team_clusters())


def device_status(workspace) -> int:
    """The decode kernel's status word from the workspace of the last step
    (0 = ok).  Reads device memory: synchronises with the workspace's stream."""
    return int(workspace[:4].view(torch.int32).item())


def mla_plan_splits(seq_lens, split_budget, stream=None):
    """Device split plan: (split_indptr [R+1] int32, chunk [1] int64)."""
    _require(seq_lens.is_cuda and seq_lens.dtype == torch.int32 and seq_lens.is_contiguous()
             and seq_lens.dim() == 1, "seq_lens must be a contiguous CUDA int32 vector")
    R = seq_lens.shape[0]
    indptr = torch.empty(R + 1, dtype=torch.int32, device=seq_lens.device)
    chunk = torch.empty(1, dtype=torch.int64, device=seq_lens.device)
    status = _native.lib().mla_plan_splits(seq_lens.data_ptr(), R, int(split_budget),
                                           indptr.data_ptr(), chunk.data_ptr(),
                                           _stream_ptr(stream, seq_lens.device))
    _native.check(status, "mla_plan_splits")
    return indptr, chunk


def mla_dcp_shard(page_table, seq_lens, world, rank, stream=None):
    """Rank `rank`'s page table and history lengths for decode context
    parallelism over `world` ranks (page column c of request r belongs to rank
    (c + r) mod world): (table_k [R, ceil(ld / world)] int32, lens_k [R] int32),
    computed on the device."""
    _require(page_table.is_cuda and page_table.dtype == torch.int32 and page_table.dim() == 2
             and page_table.stride(1) == 1, "page_table must be a CUDA int32 [R, ld] view")
    _require(seq_lens.is_cuda and seq_lens.dtype == torch.int32 and seq_lens.is_contiguous(),
             "seq_lens must be a contiguous CUDA int32 vector")
    R = seq_lens.shape[0]
    ld = page_table.stride(0)
    out_ld = max(1, -(-ld // world))
    table_k = torch.empty(R, out_ld, dtype=torch.int32, device=page_table.device)
    lens_k = torch.empty(R, dtype=torch.int32, device=page_table.device)
    _native.check(_native.lib().mla_dcp_shard(page_table.data_ptr(), ld, seq_lens.data_ptr(), R,
                                              int(world), int(rank), table_k.data_ptr(), out_ld,
                                              lens_k.data_ptr(),
                                              _stream_ptr(stream, page_table.device)),
                  "mla_dcp_shard")
    return table_k, lens_k


def mla_split_combine(o_part, lse_part, split_indptr, gate, *, n_q=1, out=None, lse=None,
                      stream=None, with_lse=True):
    """Merge chunk partials and apply the sigmoid gate; returns (out, lse)."""
    _check_bf16(gate, "gate")
    T, H, _ = gate.shape
    R = T // n_q
    rows = n_q * H
    _require(o_part.is_cuda and o_part.dtype == torch.float32 and o_part.is_contiguous()
             and o_part.dim() == 3 and o_part.shape[1:] == (rows, LATENT),
             "o_part must be contiguous CUDA fp32 [splits, n_q*H, 512]")
    _require(lse_part.is_cuda and lse_part.dtype == torch.float32 and lse_part.is_contiguous()
             and tuple(lse_part.shape) == (o_part.shape[0], rows),
             "lse_part must be contiguous CUDA fp32 [splits, n_q*H]")
    _require(split_indptr.is_cuda and split_indptr.dtype == torch.int32
             and tuple(split_indptr.shape) == (R + 1,), "split_indptr must be CUDA int32 [R+1]")
    if out is None:
        out = torch.empty_like(gate)
    if lse is None and with_lse:
        lse = torch.empty(T, H, dtype=torch.float32, device=gate.device)
    status = _native.lib().mla_split_combine(
        o_part.data_ptr(), lse_part.data_ptr(), split_indptr.data_ptr(), gate.data_ptr(), R,
        n_q, H, out.data_ptr(), lse.data_ptr() if lse is not None else None,
        _stream_ptr(stream, gate.device))
    _native.check(status, "mla_split_combine")
    return out, lse


def mla_merge_partials(out_parts, lse_parts, *, out=None, lse=None, stream=None, with_lse=True):
    """Merge the gated outputs of ranks that each decoded a disjoint part of the
    histories (decode context parallelism).  out_parts is bf16 [world, T, H, 512]
    (rank k's mla_decode output), lse_parts fp32 [world, T, H]; returns the
    merged (out [T, H, 512] bf16, lse [T, H] fp32)."""
    _require(out_parts.is_cuda and out_parts.dtype == torch.bfloat16 and out_parts.is_contiguous()
             and out_parts.dim() == 4 and out_parts.shape[-1] == LATENT,
             "out_parts must be contiguous CUDA bf16 [world, T, H, 512]")
    world, T, H, _ = out_parts.shape
    _require(lse_parts.is_cuda and lse_parts.dtype == torch.float32 and lse_parts.is_contiguous()
             and tuple(lse_parts.shape) == (world, T, H),
             "lse_parts must be contiguous CUDA fp32 [world, T, H]")
    if out is None:
        out = torch.empty(T, H, LATENT, dtype=torch.bfloat16, device=out_parts.device)
    _check_bf16(out, "out", (T, H, LATENT))
    if lse is None and with_lse:
        lse = torch.empty(T, H, dtype=torch.float32, device=out_parts.device)
    if lse is not None:
        _require(lse.is_cuda and lse.dtype == torch.float32 and lse.is_contiguous()
                 and tuple(lse.shape) == (T, H), "lse must be a contiguous CUDA fp32 [T, H]")
    status = _native.lib().mla_merge_partials(
        out_parts.data_ptr(), lse_parts.data_ptr(), world, T * H, out.data_ptr(),
        lse.data_ptr() if lse is not None else None, _stream_ptr(stream, out_parts.device))
    _native.check(status, "mla_merge_partials")
    return out, lse


def mla_kv_append_fp8(latent_new, rope_new, slab, page_table, seq_lens, n_new, *, kv_scale,
                      status=None, stream=None):
    """mla_kv_append into E4M3 pages (slab uint8 or float8_e4m3fn [num_pages,
    page_stride]): each value is stored as the E4M3 code of value / kv_scale."""
    return _append(latent_new, rope_new, _byte_view(slab), page_table, seq_lens, n_new, status,
                   stream, float(kv_scale))


def mla_kv_append(latent_new, rope_new, slab, page_table, seq_lens, n_new, *, status=None,
                  stream=None):
    """Write each request's n_new new latent / rope rows into the page pool.

    latent_new [R*n_new, 512] and rope_new [R*n_new, 64] bf16 (row r*n_new + j is
    request r's new token j); slab, page_table as for mla_decode; seq_lens [R]
    int32 histories after the append, so token j lands at position
    seq_lens[r] - n_new + j.  ``status``: optional CUDA int32 tensor of one
    element that the kernel sets to 32 (a history shorter than n_new) or 33 (a
    page ID outside the pool); such rows are skipped.  Asynchronous.
    """
    return _append(latent_new, rope_new, slab, page_table, seq_lens, n_new, status, stream,
                   None)


def _append(latent_new, rope_new, slab, page_table, seq_lens, n_new, status, stream, kv_scale):
    fp8 = kv_scale is not None
    R = int(seq_lens.shape[0]) if hasattr(seq_lens, "shape") else 0
    _require(seq_lens.is_cuda and seq_lens.dtype == torch.int32 and seq_lens.is_contiguous()
             and seq_lens.dim() == 1, "seq_lens must be a contiguous CUDA int32 vector")
    _check_bf16(latent_new, "latent_new", (R * n_new, 512))
    _check_bf16(rope_new, "rope_new", (R * n_new, 64))
    want = torch.uint8 if fp8 else torch.bfloat16
    _require(slab.is_cuda and slab.dtype == want and slab.dim() == 2 and slab.stride(1) == 1,
             f"slab must be a CUDA {want} [num_pages, page_stride] view")
    _require(slab.shape[1] >= PAGE_TOKENS * ROW, "slab page too small")
    _require(page_table.is_cuda and page_table.dtype == torch.int32 and page_table.dim() == 2
             and page_table.shape[0] == R and page_table.stride(1) == 1,
             "page_table must be a CUDA int32 [R, >= pages] view with unit column stride")
    if status is not None:
        _require(status.is_cuda and status.dtype == torch.int32 and status.numel() >= 1,
                 "status must be a CUDA int32 tensor")
    lib = _native.lib()
    head = (latent_new.data_ptr(), rope_new.data_ptr(), slab.data_ptr(), slab.shape[0],
            slab.stride(0))
    tail = (page_table.data_ptr(), page_table.stride(0), seq_lens.data_ptr(), R, int(n_new),
            None if status is None else status.data_ptr(), _stream_ptr(stream, slab.device))
    if fp8:
        rc = lib.mla_kv_append_fp8(*head, kv_scale, *tail)
    else:
        rc = lib.mla_kv_append(*head, *tail)
    _native.check(rc, "mla_kv_append_fp8" if fp8 else "mla_kv_append")
