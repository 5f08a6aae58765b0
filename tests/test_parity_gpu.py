"""GPU parity: the CUDA path (through the C ABI) against the double-precision oracle.

Bar: |out - ref| <= 1e-2 + 1e-2 |ref| on the bf16 output, |lse - ref| <= 1e-3 on
the fp32 log-sum-exp, page indexing bit-exact (one-hot probes), integer plans
bit-exact, and bit-identical results under page permutation and across runs.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from helpers import (SCALE, assert_parity, gpu_decode, oracle_decode, sample_rows,
                     to_device)
from paged_latent_attention_gb300 import api, inputs

pytestmark = pytest.mark.gpu


def _problem(lengths, n_q, H, seed, spare=3, table_ld=None, page_pad=0, poison=True):
    w = inputs.custom_workload(lengths, n_q, H, seed=seed, spare_pages=spare, table_ld=table_ld,
                               page_stride=inputs.PAGE_TOKENS * inputs.ROW_ELEMS + page_pad)
    qn, qr, gate = inputs.make_queries(w, "cpu")
    slab = inputs.make_slab(w, "cpu", poison_nan=poison)
    return w, qn, qr, gate, slab


# --------------------------------------------------------------------------
# small cases: several tiles, ragged tails, NaN-poisoned tails and free pages
# --------------------------------------------------------------------------

def test_tiny_workload_all_rows():
    w = inputs.make_workload("tiny")
    qn, qr, gate = inputs.make_queries(w, "cpu")
    slab = inputs.make_slab(w, "cpu", poison_nan=True)
    d = to_device(w, qn, qr, gate, slab)
    out, lse = gpu_decode(w, d)
    ref_out, ref_lse = oracle_decode(w, qn, qr, gate, slab)
    assert_parity(out, lse, ref_out, ref_lse, what="tiny")


RAGGED = [1, 2, 127, 128, 129, 1535, 1536, 1537, 4099]


@pytest.mark.parametrize("n_q,H", [(1, 16), (1, 64), (4, 16), (4, 64), (1, 128), (3, 16)])
@pytest.mark.parametrize("cta_budget,min_splits", [(0, 1), (4, 1), (0, 9)])
def test_ragged_histories(n_q, H, cta_budget, min_splits):
    w, qn, qr, gate, slab = _problem(RAGGED, n_q, H, seed=100 + n_q * 7 + H)
    d = to_device(w, qn, qr, gate, slab)
    out, lse = gpu_decode(w, d, cta_budget=cta_budget, min_splits=min_splits)
    ref_out, ref_lse = oracle_decode(w, qn, qr, gate, slab)
    assert_parity(out, lse, ref_out, ref_lse, what=f"ragged n_q={n_q} H={H}")


def test_empty_history_gives_zero_and_minus_inf():
    w, qn, qr, gate, slab = _problem([0, 300, 0], 1, 16, seed=5)
    w.page_table[0, :] = w.page_table[1, 0]
    d = to_device(w, qn, qr, gate, slab)
    out, lse = gpu_decode(w, d)
    o = out.float().cpu().view(3, 16, 512)
    l = lse.cpu().view(3, 16)
    assert torch.all(o[0] == 0) and torch.all(o[2] == 0)
    assert torch.all(torch.isneginf(l[0])) and torch.all(torch.isneginf(l[2]))
    ref_out, ref_lse = oracle_decode(w, qn, qr, gate, slab)
    assert_parity(out, lse, ref_out, ref_lse, what="empty")


def test_strided_page_table_view():
    """The table's row stride is honoured: a column slice of a wider table whose
    extra columns point at NaN-filled free pages."""
    w, qn, qr, gate, slab = _problem([3000, 5000, 200], 1, 64, seed=6, spare=4)
    wide = np.full((w.num_reqs, w.page_table.shape[1] + 5), 0, dtype=np.int32)
    free = sorted(set(range(w.num_pages)) - set(w.page_table[:, :].ravel().tolist()))
    wide[:, :] = free[0]
    wide[:, 2:2 + w.page_table.shape[1]] = w.page_table
    d = to_device(w, qn, qr, gate, slab)
    d["table"] = torch.as_tensor(wide, device="cuda")[:, 2:2 + w.page_table.shape[1]]
    assert not d["table"].is_contiguous()
    out, lse = gpu_decode(w, d)
    ref_out, ref_lse = oracle_decode(w, qn, qr, gate, slab)
    assert_parity(out, lse, ref_out, ref_lse, what="strided table")


def test_padded_page_stride():
    w, qn, qr, gate, slab = _problem([1600, 4000], 1, 64, seed=7, page_pad=72)
    assert w.page_stride > inputs.PAGE_TOKENS * inputs.ROW_ELEMS
    d = to_device(w, qn, qr, gate, slab)
    out, lse = gpu_decode(w, d)
    ref_out, ref_lse = oracle_decode(w, qn, qr, gate, slab)
    assert_parity(out, lse, ref_out, ref_lse, what="padded stride")


# --------------------------------------------------------------------------
# exactness probes and invariants
# --------------------------------------------------------------------------

def test_one_hot_probe_is_bit_exact_for_every_page_boundary():
    """q_rope = 2^14 e_5, one token with rope key e_5, gate logits +100 (sigmoid = 1
    exactly in fp32): the output must equal that token's latent row bit for bit."""
    page = inputs.PAGE_TOKENS
    L = 3 * page + 17
    w, qn, qr, gate, slab = _problem([L, 700], 1, 16, seed=8, spare=3)
    pages = slab.view(w.num_pages, page, 576)
    pages[..., 512:] = 0
    qn.zero_()
    qr.zero_()
    qr[:, :, 5] = 2.0 ** 14
    gate.fill_(100.0)
    d = to_device(w, qn, qr, gate, slab)
    for t_star in [0, 1, page - 1, page, 2 * page - 1, 2 * page, 3 * page - 1, 3 * page, L - 1]:
        p = int(w.page_table[0, t_star // page])
        d["slab"].view(w.num_pages, page, 576)[..., 512 + 5] = 0
        d["slab"].view(w.num_pages, page, 576)[p, t_star % page, 512 + 5] = 1.0
        for budget, min_splits in [(0, 1), (0, 16)]:
            out, lse = gpu_decode(w, d, cta_budget=budget, min_splits=min_splits)
            row = d["slab"].view(w.num_pages, page, 576)[p, t_star % page, :512]
            assert torch.equal(out[0].view(16, 512), row.expand(16, 512)), (t_star, min_splits)
            assert torch.allclose(lse[0], torch.full_like(lse[0], SCALE * 2.0 ** 14), atol=1e-3)


def test_page_permutation_and_reruns_are_bit_identical():
    w, qn, qr, gate, slab = _problem([5000, 1537, 9000], 1, 64, seed=9, spare=6)
    d = to_device(w, qn, qr, gate, slab)
    out1, lse1 = gpu_decode(w, d)
    out1b, lse1b = gpu_decode(w, d)
    assert torch.equal(out1, out1b) and torch.equal(lse1, lse1b)
    perm = np.random.Generator(np.random.PCG64(3)).permutation(w.num_pages)
    slab2 = torch.empty_like(d["slab"])
    slab2[torch.as_tensor(perm, device="cuda")] = d["slab"]
    d2 = dict(d, slab=slab2,
              table=torch.as_tensor(perm[w.page_table].astype(np.int32), device="cuda"))
    out2, lse2 = gpu_decode(w, d2)
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_split_and_unsplit_agree():
    w, qn, qr, gate, slab = _problem([20000, 7000], 1, 64, seed=10)
    d = to_device(w, qn, qr, gate, slab)
    ref_out, ref_lse = oracle_decode(w, qn, qr, gate, slab)
    for budget, min_splits in [(2, 1), (0, 1), (0, 40)]:
        out, lse = gpu_decode(w, d, cta_budget=budget, min_splits=min_splits)
        assert_parity(out, lse, ref_out, ref_lse, what=f"budget={budget} min={min_splits}")


@pytest.mark.parametrize("min_splits", [1, 4])
def test_largest_batch_of_1024_requests(min_splits):
    """The planner's request limit: 1,024 requests (four per planner thread), short
    ragged histories including empty ones, 4,096 chunks when each request must
    get 4 (the planner's chunk limit)."""
    rng = np.random.Generator(np.random.PCG64(12))
    lengths = rng.integers(0, 1500, size=1024)       # one page each: a 1.8 GB pool
    lengths[::97] = 0
    lengths[5] = 1
    w, qn, qr, gate, slab = _problem(lengths.tolist(), 1, 16, seed=12, spare=4)
    d = to_device(w, qn, qr, gate, slab)
    out, lse = gpu_decode(w, d, min_splits=min_splits)
    rows = np.concatenate([np.arange(0, 1024 * 16, 7), [1024 * 16 - 1]])
    ref_out, ref_lse = oracle_decode(w, qn, qr, gate, slab, rows=rows)
    assert_parity(out, lse, ref_out, ref_lse, rows=rows, what=f"1024 requests min={min_splits}")


def test_causal_drafts_match_single_token_runs():
    lengths = [3000, 130]
    w, qn, qr, gate, slab = _problem(lengths, 4, 16, seed=11)
    d = to_device(w, qn, qr, gate, slab)
    out4, lse4 = gpu_decode(w, d)
    for r, L in enumerate(lengths):
        for j in range(4):
            t = r * 4 + j
            w1 = inputs.Workload("one", 1, 1, 16, np.array([L - 3 + j], np.int32),
                                 w.page_table[r:r + 1], w.num_pages)
            d1 = dict(d, qn=d["qn"][t:t + 1].contiguous(), qr=d["qr"][t:t + 1].contiguous(),
                      gate=d["gate"][t:t + 1].contiguous(),
                      table=d["table"][r:r + 1].contiguous(),
                      lens=torch.tensor([L - 3 + j], dtype=torch.int32, device="cuda"))
            out1, lse1 = gpu_decode(w1, d1)
            torch.testing.assert_close(out4[t].float(), out1[0].float(), atol=1e-2, rtol=1e-2)
            torch.testing.assert_close(lse4[t], lse1[0], atol=1e-3, rtol=0)


def test_pool_above_4_gib_uses_64_bit_offsets():
    """Pages at the top of a 4.4 GB pool: element offsets exceed 2^31 and 2^32."""
    num_pages = 2500
    stride = inputs.PAGE_TOKENS * inputs.ROW_ELEMS
    assert (num_pages - 1) * stride * 2 > 4 * 2 ** 30
    lengths = [4000, 2000]
    table = np.array([[2499, 2430, 2488], [2497, 2431, 0]], dtype=np.int32)
    w = inputs.Workload("big", 2, 1, 64, np.array(lengths, np.int32), table, num_pages, seed=12)
    qn, qr, gate = inputs.make_queries(w, "cuda")
    slab = torch.full((num_pages, stride), float("nan"), dtype=torch.bfloat16, device="cuda")
    used = sorted({2499, 2430, 2488, 2497, 2431})
    g = torch.Generator(device="cuda").manual_seed(12)
    for p in used:
        slab[p].normal_(generator=g)
    # NaN tails inside the last pages stay NaN
    slab[2488, (4000 - 3072) * 576:] = float("nan")
    slab[2431, (2000 - 1536) * 576:] = float("nan")
    d = dict(qn=qn, qr=qr, gate=gate, slab=slab, table=torch.as_tensor(table, device="cuda"),
             lens=torch.as_tensor(w.seq_lens, device="cuda"))
    out, lse = gpu_decode(w, d)
    host = torch.zeros((num_pages, stride), dtype=torch.bfloat16)
    for p in used:
        host[p] = slab[p].cpu()
    ref_out, ref_lse = oracle_decode(w, qn.cpu(), qr.cpu(), gate.cpu(), host)
    assert_parity(out, lse, ref_out, ref_lse, what="4 GiB pool")
    del slab, host
    torch.cuda.empty_cache()


# --------------------------------------------------------------------------
# planner and combine, each through its own C-ABI entry point
# --------------------------------------------------------------------------

def test_plan_matches_oracle_planner():
    golden = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                         "planner_fig4.json")))["cases"]
    cases = [(c["seq_lens"], c["budget"]) for c in golden]
    rng = np.random.Generator(np.random.PCG64(20))
    for _ in range(60):
        R = int(rng.integers(1, 1025))
        lens = rng.integers(0, 1_000_001, size=R)
        lens[rng.random(R) < 0.1] = 0
        cases.append((lens.tolist(), int(rng.integers(1, 2000))))
    cases.append(([1_000_000] * 4, 608))
    cases.append(([0] * 5, 7))
    # budgets up to the library's cap (104 chunks per CTA on 152 SMs, and the limit)
    for budget in (104 * 152, 32768):
        cases.append((rng.integers(0, 1_000_001, size=64).tolist(), budget))
        cases.append(([1_000_000] * 4, budget))
    for lens, budget in cases:
        chunk, splits = oracle.plan_splits(lens, budget, 128)
        indptr, dchunk = api.mla_plan_splits(torch.tensor(lens, dtype=torch.int32,
                                                          device="cuda"), budget)
        expect = np.concatenate([[0], np.cumsum(splits)]).astype(np.int64)
        assert int(dchunk.item()) == chunk, (len(lens), budget)
        assert np.array_equal(indptr.cpu().numpy().astype(np.int64), expect)


@pytest.mark.parametrize("n_q,H", [(1, 16), (4, 64)])
def test_combine_matches_oracle_merge(n_q, H):
    lengths = [3000, 40, 7000]
    w, qn, qr, gate, slab = _problem(lengths, n_q, H, seed=13)
    chunks = [[0, 1000, 2500, 3000], [0, 40], [0, 128, 6000, 7000]]
    o_parts, l_parts, indptr = [], [], [0]
    rows_per_req = n_q * H
    for r, edges in enumerate(chunks):
        rows = np.arange(r * rows_per_req, (r + 1) * rows_per_req)
        for a, b in zip(edges[:-1], edges[1:]):
            o, l = oracle.attend_rows(qn, qr, slab, w.page_table, w.seq_lens, n_q, H, SCALE,
                                      num_pages=w.num_pages, rows=rows, t_lo=a, t_hi=b)
            o_parts.append(o)
            l_parts.append(l)
        indptr.append(indptr[-1] + len(edges) - 1)
    o_part = torch.tensor(np.stack(o_parts), dtype=torch.float32, device="cuda")
    l_part = torch.tensor(np.stack(l_parts), dtype=torch.float32, device="cuda")
    out, lse = api.mla_split_combine(o_part, l_part,
                                     torch.tensor(indptr, dtype=torch.int32, device="cuda"),
                                     gate.cuda(), n_q=n_q)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle_decode(w, qn, qr, gate, slab)
    assert_parity(out, lse, ref_out, ref_lse, what="combine")


# --------------------------------------------------------------------------
# full-size workloads, checked on sampled rows
# --------------------------------------------------------------------------

def _head_rows(w, heads):
    """Rows (token, head) for every query token and the listed heads."""
    return np.array([t * w.num_heads + h for t in range(w.num_tokens) for h in heads],
                    dtype=np.int64)


# head sets: both 32-column halves of every 64-row team (heads 0-31 and 32-63), their edges
# and a few inside; every draft token of the 4-draft workload is its own team
@pytest.mark.parametrize("name,heads", [("steady", (0, 5, 17, 31, 32, 44, 58, 63)),
                                        ("agentic", (0, 13, 31, 32, 47, 63)),
                                        ("spec", (0, 9, 31, 32, 54, 63))])
def test_workload_parity_sampled(name, heads):
    w = inputs.make_workload(name)
    qn, qr, gate = inputs.make_queries(w, "cuda")
    slab = inputs.make_slab(w, "cuda")
    d = dict(qn=qn, qr=qr, gate=gate, slab=slab,
             table=torch.as_tensor(w.page_table, device="cuda"),
             lens=torch.as_tensor(w.seq_lens, device="cuda"))
    out, lse = gpu_decode(w, d)
    rows = _head_rows(w, heads)
    host = slab.cpu()
    ref_out, ref_lse = oracle_decode(w, qn.cpu(), qr.cpu(), gate.cpu(), host, rows=rows)
    assert_parity(out, lse, ref_out, ref_lse, rows=rows, what=name)
    assert torch.isfinite(lse).all() and torch.isfinite(out.float()).all()
    del slab, host, d
    torch.cuda.empty_cache()


def test_long_context_all_24_layers():
    """4 x 1M-token histories, 24 slabs sharing one page table, >= 128 splits per
    request; every layer is checked against the oracle on 4 heads of every request
    (a different head set per layer, 96 heads over the step), and every row of every
    layer for finiteness and a plausible log-sum-exp."""
    w = inputs.make_workload("long")
    table = torch.as_tensor(w.page_table, device="cuda")
    lens = torch.as_tensor(w.seq_lens, device="cuda")
    assert api.mla_split_budget(4, 1, 64, 0, w.min_splits) >= 4 * 128
    slabs = [inputs.make_slab(w, "cuda", layer=l) for l in range(w.num_slabs)]
    queries = [inputs.make_queries(w, "cuda", layer=l) for l in range(w.num_slabs)]
    outs = []
    for l in range(w.num_slabs):
        qn, qr, gate = queries[l]
        out, lse = gpu_decode(w, dict(qn=qn, qr=qr, gate=gate, slab=slabs[l], table=table,
                                      lens=lens))
        outs.append((out, lse))
    for l, (out, lse) in enumerate(outs):
        assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all(), l
        assert float(lse.min()) > math.log(1e6) - 1 and float(lse.max()) < math.log(1e6) + 6
    rng = np.random.Generator(np.random.PCG64(24))
    for l in range(w.num_slabs):
        heads = sorted({int(rng.integers(0, 32)), int(rng.integers(32, 64)), 4 * l % 64, 63 - l})
        rows = np.array([r * 64 + h for r in range(4) for h in heads], dtype=np.int64)
        qn, qr, gate = queries[l]
        host = slabs[l].cpu()
        ref_out, ref_lse = oracle_decode(w, qn.cpu(), qr.cpu(), gate.cpu(), host, rows=rows)
        assert_parity(outs[l][0], outs[l][1], ref_out, ref_lse, rows=rows, what=f"layer {l}")
        del host
    del slabs, queries, outs
    torch.cuda.empty_cache()
