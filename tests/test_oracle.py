"""Pins for the double-precision oracle (CPU only).

Each test ties the oracle to something other than itself: a library attention
routine, the absorbed/un-absorbed MLA identity, closed forms, bit-exact probes of
the page indexing, and invariants of the definition.  A last group plants
plausible mistakes in the oracle's inputs and checks that the pins catch them.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from paged_latent_attention_gb300 import inputs

SCALE = 1.0 / math.sqrt(192.0)


def _bf16(x):
    return torch.as_tensor(x, dtype=torch.float64).to(torch.bfloat16)


def _f64(t):
    return t.to(torch.float64).numpy()


def _random_problem(seed, lengths, n_q, H, dc, dr, page_tokens, spare=3, table_ld=None,
                    page_pad=0):
    g = torch.Generator().manual_seed(seed)
    w = inputs.custom_workload(lengths, n_q, H, seed=seed, spare_pages=spare,
                               page_tokens=page_tokens, dc=dc, dr=dr, table_ld=table_ld,
                               page_stride=page_tokens * (dc + dr) + page_pad)
    T = len(lengths) * n_q
    qn = torch.randn(T, H, dc, generator=g).to(torch.bfloat16)
    qr = torch.randn(T, H, dr, generator=g).to(torch.bfloat16)
    gate = torch.randn(T, H, dc, generator=g).to(torch.bfloat16)
    slab = torch.randn(w.num_pages, w.page_stride, generator=g).to(torch.bfloat16)
    return w, qn, qr, gate, slab


def _run(w, qn, qr, gate, slab, scale=SCALE, **kw):
    return oracle.mla_decode_reference(qn, qr, gate, slab, w.page_table, w.seq_lens, w.n_q,
                                       w.num_heads, scale, num_pages=w.num_pages,
                                       page_stride=w.page_stride, page_tokens=w.page_tokens,
                                       dc=w.dc, dr=w.dr, **kw)


def _gather(w, slab, r):
    """Rows of request r in logical order (plain indexing through the table)."""
    L = int(w.seq_lens[r])
    pages = slab.view(w.num_pages, w.page_stride)[:, :w.page_tokens * (w.dc + w.dr)]
    pages = pages.reshape(w.num_pages, w.page_tokens, w.dc + w.dr)
    t = np.arange(L)
    return pages[torch.as_tensor(w.page_table[r, t // w.page_tokens].astype(np.int64)),
                 torch.as_tensor(t % w.page_tokens)]


def _sdpa_reference(w, qn, qr, gate, slab, scale=SCALE):
    """torch's scaled_dot_product_attention (float64) on contiguously gathered rows."""
    R, n_q, H, dc = w.num_reqs, w.n_q, w.num_heads, w.dc
    out = np.zeros((R * n_q * H, dc))
    lse = np.zeros(R * n_q * H)
    for r in range(R):
        x = _gather(w, slab, r).to(torch.float64)          # [L, dc+dr]
        L = x.shape[0]
        k = x                                               # keys: [c | k_rope]
        v = x[:, :dc]                                       # values: c
        q = torch.cat([qn[r * n_q:(r + 1) * n_q], qr[r * n_q:(r + 1) * n_q]], dim=-1)
        q = q.to(torch.float64).permute(1, 0, 2)            # [H, n_q, dc+dr]
        j = torch.arange(n_q)[:, None]
        t = torch.arange(L)[None, :]
        mask = t < (L - (n_q - 1 - j))                      # [n_q, L]
        o = torch.nn.functional.scaled_dot_product_attention(
            q, k.expand(H, L, -1), v.expand(H, L, -1), attn_mask=mask, scale=scale)
        s = (q @ k.T) * scale
        s = s.masked_fill(~mask, -math.inf)
        l = torch.logsumexp(s, dim=-1)                      # [H, n_q]
        g = gate[r * n_q:(r + 1) * n_q].to(torch.float64).permute(1, 0, 2)
        o = torch.sigmoid(g) * o
        rows = slice(r * n_q * H, (r + 1) * n_q * H)
        out[rows] = o.permute(1, 0, 2).reshape(-1, dc).numpy()
        lse[rows] = l.permute(1, 0).reshape(-1).numpy()
    return out, lse


# --------------------------------------------------------------------------
# library pin: torch SDPA over contiguous rows
# --------------------------------------------------------------------------

@pytest.mark.parametrize("page_tokens,n_q,H,dc,dr,lengths", [
    (1, 1, 2, 16, 8, [1, 7, 13]),
    (3, 1, 4, 32, 8, [5, 9, 40]),
    (4, 4, 2, 16, 4, [4, 11, 33]),
    (3, 4, 3, 8, 4, [6, 17]),
    (1536, 1, 4, 512, 64, [1, 200, 1537]),
])
def test_matches_library_attention(page_tokens, n_q, H, dc, dr, lengths):
    w, qn, qr, gate, slab = _random_problem(11, lengths, n_q, H, dc, dr, page_tokens)
    out, lse = _run(w, qn, qr, gate, slab)
    ref_out, ref_lse = _sdpa_reference(w, qn, qr, gate, slab)
    np.testing.assert_allclose(out, ref_out, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# textbook identity: absorbed latent attention == un-absorbed multi-head attention
# --------------------------------------------------------------------------

def test_absorbed_equals_unabsorbed_mha():
    """q_nope . (c W_UK) == (W_UK q_nope) . c, and sum_t p_t (c_t W_UV) == (sum_t p_t c_t) W_UV.

    W_UK, q_nope are small integers so the absorbed query is exact in bf16."""
    rng = np.random.Generator(np.random.PCG64(5))
    dc, dr, dh, H, page_tokens = 64, 8, 16, 3, 4
    lengths = [9, 22]
    w, _, qr, gate, slab = _random_problem(12, lengths, 1, H, dc, dr, page_tokens)
    W_UK = rng.integers(-1, 2, size=(H, dc, dh)).astype(np.float64)
    W_UV = rng.standard_normal((H, dc, dh))
    q_nope = rng.integers(-2, 3, size=(len(lengths), H, dh)).astype(np.float64)
    q_abs = np.einsum("hcd,rhd->rhc", W_UK, q_nope)        # |q_abs| <= 32: exact in bf16
    qn = _bf16(q_abs)
    assert np.array_equal(_f64(qn), q_abs)
    o_latent, lse = oracle.attend_rows(qn, qr, slab, w.page_table, w.seq_lens, 1, H, SCALE,
                                       num_pages=w.num_pages, page_stride=w.page_stride,
                                       page_tokens=page_tokens, dc=dc, dr=dr)
    o_latent = o_latent.reshape(len(lengths), H, dc)
    for r in range(len(lengths)):
        x = _f64(_gather(w, slab, r))
        c, k_rope = x[:, :dc], x[:, dc:]
        for h in range(H):
            k_nope = c @ W_UK[h]                           # per-token key, [L, dh]
            v = c @ W_UV[h]                                # per-token value, [L, dh]
            keys = np.concatenate([k_nope, k_rope], axis=1)
            q = np.concatenate([q_nope[r, h], _f64(qr[r, h])])
            s = SCALE * (keys @ q)
            p = scipy.special.softmax(s)
            mha = p @ v
            np.testing.assert_allclose(o_latent[r, h] @ W_UV[h], mha, rtol=1e-12, atol=1e-12)
            assert abs(lse[r * H + h] - scipy.special.logsumexp(s)) < 1e-12


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------

def test_single_token_history_is_gated_latent():
    w, qn, qr, gate, slab = _random_problem(3, [1, 1], 1, 4, 512, 64, 1536)
    out, lse = _run(w, qn, qr, gate, slab)
    for r in range(2):
        x = _f64(_gather(w, slab, r))[0]
        for h in range(4):
            row = r * 4 + h
            sig = 1.0 / (1.0 + np.exp(-_f64(gate[r, h])))
            assert np.array_equal(out[row], x[:512] / (1.0 + np.exp(-_f64(gate[r, h]))))
            np.testing.assert_allclose(out[row], sig * x[:512], rtol=1e-15, atol=0)
            s0 = SCALE * (_f64(qn[r, h]) @ x[:512] + _f64(qr[r, h]) @ x[512:])
            assert abs(lse[row] - s0) <= 1e-12 * max(1.0, abs(s0))


def test_equal_scores_give_mean_latent_and_log_length():
    lengths = [1, 2, 1536, 3001]
    w, qn, qr, gate, slab = _random_problem(4, lengths, 1, 2, 512, 64, 1536)
    qn.zero_()
    qr.zero_()
    out, lse = _run(w, qn, qr, gate, slab)
    for r, L in enumerate(lengths):
        mean = _f64(_gather(w, slab, r))[:, :512].mean(axis=0)
        for h in range(2):
            row = r * 2 + h
            np.testing.assert_allclose(out[row], scipy.special.expit(_f64(gate[r, h])) * mean,
                                       rtol=1e-12, atol=1e-13)
            assert abs(lse[row] - math.log(L)) < 1e-12


def test_one_hot_probe_selects_exact_row_for_every_page_boundary():
    """q_rope = 2^14 e_k and a single token whose rope key is e_k: the softmax
    weight of every other token underflows to exactly 0 in double, so the output
    is exactly sigma(g) * c_{t*}.  Probes the first/last row of each page and the
    last row of a partial page."""
    page_tokens = 1536
    lengths = [3 * page_tokens + 17]
    w, qn, qr, gate, slab = _random_problem(5, lengths, 1, 1, 512, 64, page_tokens, spare=4)
    L = lengths[0]
    probes = [0, 1, page_tokens - 1, page_tokens, 2 * page_tokens - 1, 2 * page_tokens,
              3 * page_tokens - 1, 3 * page_tokens, L - 1]
    pages = slab.view(w.num_pages, page_tokens, 576)
    pages[..., 512:] = 0
    qn.zero_()
    qr.zero_()
    qr[0, 0, 5] = 2.0 ** 14
    for t_star in probes:
        p = int(w.page_table[0, t_star // page_tokens])
        pages[..., 512 + 5] = 0
        pages[p, t_star % page_tokens, 512 + 5] = 1.0
        out, lse = _run(w, qn, qr, gate, slab)
        c = _f64(pages[p, t_star % page_tokens, :512])
        expect = c / (1.0 + np.exp(-_f64(gate[0, 0])))
        assert np.array_equal(out[0], expect), t_star
        assert lse[0] == pytest.approx(SCALE * 2.0 ** 14, abs=1e-9)


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------

def test_page_permutation_is_bit_identical():
    w, qn, qr, gate, slab = _random_problem(6, [700, 3100, 1536], 1, 4, 512, 64, 1536, spare=5)
    out, lse = _run(w, qn, qr, gate, slab)
    perm = np.random.Generator(np.random.PCG64(9)).permutation(w.num_pages)
    slab2 = torch.empty_like(slab)
    slab2[torch.as_tensor(perm)] = slab          # physical page p moves to perm[p]
    w.page_table = perm[w.page_table].astype(np.int32)
    out2, lse2 = _run(w, qn, qr, gate, slab2)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


@pytest.mark.parametrize("bounds", [[0, 128, 1024], [0, 1536, 3072], [0, 1, 2, 5000],
                                    [0, 7, 640, 641, 2000]])
def test_split_then_merge_equals_unsplit(bounds):
    w, qn, qr, gate, slab = _random_problem(7, [2000, 33, 640], 1, 4, 512, 64, 1536)
    o_full, lse_full = oracle.attend_rows(qn, qr, slab, w.page_table, w.seq_lens, 1, 4, SCALE,
                                          num_pages=w.num_pages)
    edges = bounds + [10 ** 9]
    parts = [oracle.attend_rows(qn, qr, slab, w.page_table, w.seq_lens, 1, 4, SCALE,
                                num_pages=w.num_pages, t_lo=a, t_hi=b)
             for a, b in zip(edges[:-1], edges[1:])]
    o, lse = oracle.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    np.testing.assert_allclose(o, o_full, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, lse_full, rtol=1e-13, atol=1e-13)


def test_merge_matches_library_logsumexp_and_handles_empty_chunks():
    rng = np.random.Generator(np.random.PCG64(8))
    lse_parts = rng.standard_normal((5, 7)) * 4
    lse_parts[1, :] = -np.inf                     # an empty chunk
    lse_parts[:, 3] = -np.inf                     # a row no chunk reaches
    o_parts = rng.standard_normal((5, 7, 6))
    o, lse = oracle.lse_merge(o_parts, lse_parts)
    for row in range(7):
        if row == 3:
            assert lse[row] == -np.inf and not o[row].any()
            continue
        assert abs(lse[row] - scipy.special.logsumexp(lse_parts[:, row])) < 1e-13
        wts = scipy.special.softmax(lse_parts[:, row])
        np.testing.assert_allclose(o[row], wts @ o_parts[:, row], rtol=1e-13, atol=1e-14)


def test_causal_drafts_equal_shorter_single_token_runs():
    lengths = [50, 1539, 4]
    n_q, H = 4, 3
    w, qn, qr, gate, slab = _random_problem(9, lengths, n_q, H, 512, 64, 1536)
    out, lse = _run(w, qn, qr, gate, slab)
    for r, L in enumerate(lengths):
        for j in range(n_q):
            w1 = inputs.Workload("one", 1, 1, H, np.array([L - (n_q - 1 - j)], np.int32),
                                 w.page_table[r:r + 1], w.num_pages)
            t = r * n_q + j
            o1, l1 = _run(w1, qn[t:t + 1], qr[t:t + 1], gate[t:t + 1], slab)
            rows = slice(t * H, (t + 1) * H)
            assert np.array_equal(out[rows], o1) and np.array_equal(lse[rows], l1)


def test_causal_row_with_no_visible_token():
    w, qn, qr, gate, slab = _random_problem(10, [2], 4, 2, 512, 64, 1536)
    out, lse = _run(w, qn, qr, gate, slab)
    # drafts j = 0, 1 see L - 3 + j <= 0 tokens
    assert np.all(lse[:4] == -np.inf) and not out[:4].any()
    assert np.all(np.isfinite(lse[4:]))


def test_nan_poisoned_tails_and_free_pages_never_reach_output():
    w, qn, qr, gate, slab = _random_problem(13, [100, 1536, 1700], 1, 4, 512, 64, 1536,
                                            spare=3, table_ld=4, page_pad=64)
    out, lse = _run(w, qn, qr, gate, slab)
    poisoned = slab.clone()
    inputs.poison_slab(w, poisoned)
    assert torch.isnan(poisoned.float()).any()
    out2, lse2 = _run(w, qn, qr, gate, poisoned)
    assert np.all(np.isfinite(out2)) and np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_gate_is_the_logistic_sigmoid():
    x = np.linspace(-40, 40, 161)
    o = np.linspace(-3, 3, 161)
    np.testing.assert_allclose(oracle.gate_sigmoid(o, x), scipy.special.expit(x) * o,
                               rtol=1e-15, atol=1e-300)
    assert oracle.gate_sigmoid(np.array([2.0]), np.array([0.0]))[0] == 1.0


def test_out_of_pool_page_is_reported():
    w, qn, qr, gate, slab = _random_problem(14, [10], 1, 1, 16, 4, 4)
    w.page_table[0, 1] = w.num_pages
    with pytest.raises(IndexError):
        _run(w, qn, qr, gate, slab)


# --------------------------------------------------------------------------
# planted mistakes: the pins above must notice each of these
# --------------------------------------------------------------------------

def _mismatch(a, b, rtol=1e-11, atol=1e-12):
    return not np.allclose(a, b, rtol=rtol, atol=atol)


def test_planted_wrong_scale_is_caught():
    w, qn, qr, gate, slab = _random_problem(15, [40, 9], 1, 2, 32, 8, 3)
    ref_out, ref_lse = _sdpa_reference(w, qn, qr, gate, slab)
    out, lse = _run(w, qn, qr, gate, slab, scale=1.0 / math.sqrt(40.0))
    assert _mismatch(out, ref_out) and _mismatch(lse, ref_lse)


def test_planted_dropped_rope_term_is_caught():
    w, qn, qr, gate, slab = _random_problem(16, [40, 9], 1, 2, 32, 8, 3)
    ref_out, ref_lse = _sdpa_reference(w, qn, qr, gate, slab)
    out, lse = _run(w, qn, torch.zeros_like(qr), gate, slab)
    assert _mismatch(out, ref_out) and _mismatch(lse, ref_lse)


def test_planted_page_table_shift_is_caught():
    w, qn, qr, gate, slab = _random_problem(17, [40, 9], 1, 2, 32, 8, 3, spare=4)
    ref_out, _ = _sdpa_reference(w, qn, qr, gate, slab)
    w.page_table = np.roll(w.page_table, 1, axis=1)
    out, _ = _run(w, qn, qr, gate, slab)
    assert _mismatch(out, ref_out)


def test_planted_transposed_query_heads_are_caught():
    w, qn, qr, gate, slab = _random_problem(18, [40, 9], 1, 2, 32, 8, 3)
    ref_out, _ = _sdpa_reference(w, qn, qr, gate, slab)
    out, _ = _run(w, qn.flip(1).contiguous(), qr, gate, slab)
    assert _mismatch(out, ref_out)
