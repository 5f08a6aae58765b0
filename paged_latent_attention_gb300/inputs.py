"""Seeded synthetic inputs for paged gated-MLA decode.

This module holds none of the method's arithmetic: it only draws history
lengths, page assignments, pool contents, queries and gate logits from seeded
generators.  Both the CUDA path's tests/benchmark and the CPU oracle consume
what it produces, so it lives apart from both.

Workloads (history-length mixes, pool sizes and seeds):

  tiny     2 requests x 1 query token, 16 heads, histories 1000 and 2000,
           one slab of 8 pages, page IDs drawn without replacement, seed 0
  steady   64 x 1, 64 heads, histories uniform in [8192, 32768], 2048 pages
           assigned by a random permutation, seed 1
  agentic  32 x 1, 64 heads, lognormal histories with median 88k and p90 272k
           tokens (the agentic input-length spread reported for the AgentX
           trace in the AgentX - InferenceXv3 report), capped at 1,000,000;
           pool = pages needed + 10% free pages, scattered IDs, seed 2
  spec     128 x 4 query tokens (causal among the 4 drafts), 64 heads,
           histories uniform in [4096, 65536], pool = pages needed + 10%, seed 3
  long     4 x 1 at 1,000,000 tokens, 64 heads, 24 slabs (one per MLA layer)
           sharing one table of 652 pages per request, >= 128 splits per
           request, seed 4
  extend   4 requests x 128 new tokens (a chunked extend: causal among the
           new tokens, whose rows are the history's last 128), 64 heads,
           histories uniform in [8192, 32768], pool = pages needed + 10%,
           seed 5

Values: q, KV rows and gate logits are N(0, 1) rounded to bf16.  Tail rows of a
request's last page and free pages may be poisoned with NaN (reused pages can
hold stale non-finite data, vLLM Kimi K3 blog, "Correctness Risks Introduced by
Tensor Reuse"), which a correct decode never lets reach its output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

PAGE_TOKENS = 1536
DC = 512
DR = 64
ROW_ELEMS = DC + DR


@dataclass
class Workload:
    name: str
    num_reqs: int
    n_q: int
    num_heads: int
    seq_lens: np.ndarray          # int32 [R]
    page_table: np.ndarray        # int32 [R, table_ld]
    num_pages: int
    num_slabs: int = 1
    seed: int = 0
    min_splits: int = 1
    page_tokens: int = PAGE_TOKENS
    dc: int = DC
    dr: int = DR
    page_stride: int = 0          # elements between pages; 0 = page_tokens * (dc + dr)
    notes: dict = field(default_factory=dict)

    def __post_init__(self):
        if self.page_stride == 0:
            self.page_stride = self.page_tokens * (self.dc + self.dr)

    @property
    def num_tokens(self) -> int:  # query tokens T = R * n_q
        return self.num_reqs * self.n_q

    @property
    def kv_tokens(self) -> int:
        return int(np.asarray(self.seq_lens, dtype=np.int64).sum())

    @property
    def kv_bytes_per_layer(self) -> int:
        return self.kv_tokens * (self.dc + self.dr) * 2

    @property
    def visible_pairs(self) -> int:
        """(query row, KV token) pairs of one layer: draft/new token j of request
        r sees seq_lens[r] - (n_q - 1 - j) tokens, for each of the heads."""
        L = np.asarray(self.seq_lens, dtype=np.int64)
        j = np.arange(self.n_q, dtype=np.int64)
        vis = np.maximum(0, L[:, None] - (self.n_q - 1 - j[None, :]))
        return int(vis.sum()) * self.num_heads


def _pages_for(lengths, page_tokens):
    return [max(0, -(-int(L) // page_tokens)) for L in lengths]


def _assign_pages(rng, lengths, num_pages, page_tokens, table_ld=None, filler=None):
    """Scatter each request's logical pages over the pool with a random permutation."""
    need = _pages_for(lengths, page_tokens)
    total = sum(need)
    if total > num_pages:
        raise ValueError(f"pool of {num_pages} pages cannot hold {total} pages")
    perm = rng.permutation(num_pages).astype(np.int32)
    ld = table_ld or max(1, max(need) if need else 1)
    table = np.zeros((len(lengths), ld), dtype=np.int32)
    free = perm[total:]
    pos = 0
    for r, n in enumerate(need):
        table[r, :n] = perm[pos:pos + n]
        pos += n
        # entries past the request's last page are never read; point them at a
        # free page (or page 0) so an erroneous read stays inside the pool
        table[r, n:] = (free[0] if len(free) else 0) if filler is None else filler
    return table


def make_workload(name: str) -> Workload:
    """The five named workloads (see the module docstring)."""
    if name == "tiny":
        rng = np.random.Generator(np.random.PCG64(0))
        lens = np.array([1000, 2000], dtype=np.int32)
        table = _assign_pages(rng, lens, 8, PAGE_TOKENS)
        return Workload("tiny", 2, 1, 16, lens, table, 8, seed=0)
    if name == "steady":
        rng = np.random.Generator(np.random.PCG64(1))
        lens = rng.integers(8192, 32768, size=64, endpoint=True).astype(np.int32)
        table = _assign_pages(rng, lens, 2048, PAGE_TOKENS)
        return Workload("steady", 64, 1, 64, lens, table, 2048, seed=1)
    if name == "agentic":
        rng = np.random.Generator(np.random.PCG64(2))
        mu = math.log(88_000.0)
        sigma = math.log(272_000.0 / 88_000.0) / 1.2815515655446004  # z(0.9)
        lens = np.rint(rng.lognormal(mu, sigma, size=32))
        lens = np.clip(lens, 1, 1_000_000).astype(np.int32)
        need = sum(_pages_for(lens, PAGE_TOKENS))
        pages = need + -(-need // 10)
        table = _assign_pages(rng, lens, pages, PAGE_TOKENS)
        return Workload("agentic", 32, 1, 64, lens, table, pages, seed=2,
                        notes={"lognormal_mu": mu, "lognormal_sigma": sigma})
    if name == "spec":
        rng = np.random.Generator(np.random.PCG64(3))
        lens = rng.integers(4096, 65536, size=128, endpoint=True).astype(np.int32)
        need = sum(_pages_for(lens, PAGE_TOKENS))
        pages = need + -(-need // 10)
        table = _assign_pages(rng, lens, pages, PAGE_TOKENS)
        return Workload("spec", 128, 4, 64, lens, table, pages, seed=3)
    if name == "extend":
        rng = np.random.Generator(np.random.PCG64(5))
        lens = rng.integers(8192, 32768, size=4, endpoint=True).astype(np.int32)
        need = sum(_pages_for(lens, PAGE_TOKENS))
        pages = need + -(-need // 10)
        table = _assign_pages(rng, lens, pages, PAGE_TOKENS)
        return Workload("extend", 4, 128, 64, lens, table, pages, seed=5)
    if name == "long":
        rng = np.random.Generator(np.random.PCG64(4))
        lens = np.full(4, 1_000_000, dtype=np.int32)
        table = _assign_pages(rng, lens, 4 * 652, PAGE_TOKENS)
        return Workload("long", 4, 1, 64, lens, table, 4 * 652, num_slabs=24, seed=4,
                        min_splits=128)
    raise KeyError(name)


def equal_length_control(w: Workload) -> Workload:
    """The equal-length control of a workload (TokenSpeed AgentX post, section
    "Balance MLA work with per-request KV splitting", the paragraph under
    Figure 5): the same requests and the same total KV tokens, every history at
    the batch's average length (the remainder of the division spread one token
    each over the first requests); pool = pages needed + 10% free, scattered."""
    total = w.kv_tokens
    R = w.num_reqs
    lens = np.full(R, total // R, dtype=np.int64)
    lens[: total % R] += 1
    lens = lens.astype(np.int32)
    rng = np.random.Generator(np.random.PCG64([int(w.seed), 99]))
    need = sum(_pages_for(lens, w.page_tokens))
    pages = need + -(-need // 10)
    table = _assign_pages(rng, lens, pages, w.page_tokens)
    return Workload(w.name + "-control", R, w.n_q, w.num_heads, lens, table, pages,
                    num_slabs=w.num_slabs, seed=w.seed, min_splits=w.min_splits,
                    page_tokens=w.page_tokens, dc=w.dc, dr=w.dr)


WORKLOAD_NAMES = ("tiny", "steady", "agentic", "spec", "long", "extend")


def custom_workload(lengths, n_q, num_heads, *, seed=0, spare_pages=2, page_tokens=PAGE_TOKENS,
                    table_ld=None, dc=DC, dr=DR, page_stride=0, name="custom") -> Workload:
    """A small workload with explicit histories (edge cases, tests)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = np.asarray(lengths, dtype=np.int32)
    need = sum(_pages_for(lens, page_tokens))
    pages = need + spare_pages
    table = _assign_pages(rng, lens, pages, page_tokens, table_ld=table_ld)
    return Workload(name, len(lens), n_q, num_heads, lens, table, pages, seed=seed,
                    page_tokens=page_tokens, dc=dc, dr=dr, page_stride=page_stride)


# ---------------------------------------------------------------------------
# tensors (torch is used only as a seeded random source and as storage)
# ---------------------------------------------------------------------------

def _gen(device, seed):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_queries(w: Workload, device="cpu", layer: int = 0):
    """q_nope_absorbed [T, H, dc], q_rope [T, H, dr], gate logits [T, H, dc], all bf16."""
    import torch
    T, H = w.num_tokens, w.num_heads
    g = _gen(device, w.seed * 1_000_003 + layer * 101 + 7)
    qn = torch.empty(T, H, w.dc, dtype=torch.bfloat16, device=device).normal_(generator=g)
    qr = torch.empty(T, H, w.dr, dtype=torch.bfloat16, device=device).normal_(generator=g)
    gate = torch.empty(T, H, w.dc, dtype=torch.bfloat16, device=device).normal_(generator=g)
    return qn, qr, gate


def make_slab(w: Workload, device="cpu", layer: int = 0, poison_nan: bool = False,
              pages_per_chunk: int = 64):
    """One layer's slab: [num_pages, page_stride] bf16 of N(0, 1) rows.

    With ``poison_nan`` the rows past each request's history in its last page,
    every free page and any padding between pages hold NaN.
    """
    import torch
    g = _gen(device, w.seed * 1_000_003 + layer * 101 + 3)
    slab = torch.empty(w.num_pages, w.page_stride, dtype=torch.bfloat16, device=device)
    for p0 in range(0, w.num_pages, pages_per_chunk):
        p1 = min(w.num_pages, p0 + pages_per_chunk)
        slab[p0:p1].normal_(generator=g)
    if poison_nan:
        poison_slab(w, slab)
    return slab


HOST_PAGE_BANK = 16


def make_host_pages(w: Workload, req_ids, layer: int = 0, fp8: bool = False,
                    kv_scale: float = None):
    """Host pages for the listed requests, for timing the oracle on a sample of
    a workload whose pool is too large to draw on the host in reasonable time.
    HOST_PAGE_BANK pages of N(0, 1) values are drawn from numpy's PCG64 keyed by
    (seed, layer) and rounded to bf16 (or, with ``fp8``, cast to E4M3 as
    make_slab_e4m3 does); each sampled page is a copy of a bank page chosen at
    random.  The values follow the workload's recipe but are not the device
    pool's values: use this only where the result is not compared.

    Returns (slab [n_pages, page_stride] bf16 or uint8, table [len(req_ids), ld]
    int32 indexing it, seq_lens int32 [len(req_ids)])."""
    import torch
    rng = np.random.Generator(np.random.PCG64([int(w.seed), int(layer), 17]))
    per = [-(-int(w.seq_lens[r]) // w.page_tokens) for r in req_ids]
    n = max(1, sum(per))
    bank = torch.from_numpy(rng.standard_normal((HOST_PAGE_BANK, w.page_stride),
                                                dtype=np.float32))
    if fp8:
        scale = KV_SCALE_E4M3 if kv_scale is None else kv_scale
        bank = bank.div_(scale).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    else:
        bank = bank.to(torch.bfloat16)
    pick = torch.from_numpy(rng.integers(0, HOST_PAGE_BANK, size=n))
    slab = bank.index_select(0, pick)
    table = np.zeros((len(req_ids), max(1, max(per) if per else 1)), dtype=np.int32)
    pos = 0
    for i, k in enumerate(per):
        table[i, :k] = np.arange(pos, pos + k)
        pos += k
    lens = np.asarray([int(w.seq_lens[r]) for r in req_ids], dtype=np.int32)
    return slab, table, lens


# Scale of the synthetic FP8 cache: N(0, 1) values reach E4M3's largest finite
# value (448) at 6 standard deviations.
KV_SCALE_E4M3 = 6.0 / 448.0
E4M3_NAN = 0x7F


def make_slab_e4m3(w: Workload, device="cpu", layer: int = 0, poison_nan: bool = False,
                   kv_scale: float = KV_SCALE_E4M3, pages_per_chunk: int = 64):
    """One layer's FP8 slab: [num_pages, page_stride] uint8 holding E4M3 bytes of
    N(0, 1) / kv_scale (clamped to +-448), made with torch's float8_e4m3fn cast
    from the same seeded stream as make_slab.  page_stride counts bytes here.
    With ``poison_nan`` the bytes a decode must not read hold the E4M3 NaN."""
    import torch
    g = _gen(device, w.seed * 1_000_003 + layer * 101 + 3)
    slab = torch.empty(w.num_pages, w.page_stride, dtype=torch.uint8, device=device)
    for p0 in range(0, w.num_pages, pages_per_chunk):
        p1 = min(w.num_pages, p0 + pages_per_chunk)
        vals = torch.empty(p1 - p0, w.page_stride, dtype=torch.float32, device=device)
        vals.normal_(generator=g)
        vals.div_(kv_scale).clamp_(-448.0, 448.0)
        slab[p0:p1] = vals.to(torch.float8_e4m3fn).view(torch.uint8)
        del vals
    if poison_nan:
        poison_slab(w, slab, value=E4M3_NAN)
    return slab


def poison_slab(w: Workload, slab, value=None):
    """Write NaN (or ``value``, e.g. the E4M3 NaN byte) into every slab element a
    decode must not read."""
    import torch
    nan = float("nan") if value is None else value
    used_rows = w.page_tokens * (w.dc + w.dr)
    if w.page_stride > used_rows:
        slab[:, used_rows:] = nan
    need = _pages_for(w.seq_lens, w.page_tokens)
    used = set()
    for r, n in enumerate(need):
        pages = [int(p) for p in w.page_table[r, :n]]
        used.update(pages)
        L = int(w.seq_lens[r])
        if n and L % w.page_tokens:
            last = pages[-1]
            tail0 = (L % w.page_tokens) * (w.dc + w.dr)
            slab[last, tail0:used_rows] = nan
    free = [p for p in range(w.num_pages) if p not in used]
    if free:
        idx = torch.tensor(free, dtype=torch.long, device=slab.device)
        slab.index_fill_(0, idx, nan)
    return slab
