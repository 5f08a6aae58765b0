"""Pins for the oracle's KV append (CPU only).

The append-only contract (vLLM blog "Kimi K3 Inference Backend Evolution",
section "State Overwrite: How KDA Breaks Traditional KV Cache"): a new token's
rows go after the request's history and no earlier row changes.  The checks
below tie the oracle to plain constructions: where each row lands in the pool
(brute force over small pages), that appending token by token builds the same
pool as writing the history at once, and that decoding the appended pool is the
softmax over the explicit list of rows.
"""
import numpy as np
import pytest

import oracle

DC, DR = 8, 4          # small rows so brute force stays readable
ROW = DC + DR


def _bf16_bits(x):
    """float -> bf16 bit patterns (round to nearest even), as uint16."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def _bits_to_f64(b):
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def _rows(rng, n):
    return _bf16_bits(rng.standard_normal((n, DC))), _bf16_bits(rng.standard_normal((n, DR)))


def test_rows_land_at_their_page_and_offset_and_nothing_else_changes():
    rng = np.random.Generator(np.random.PCG64(1))
    page_tokens, num_pages = 4, 9
    slab = _bf16_bits(rng.standard_normal((num_pages, page_tokens * ROW)))
    table = np.array([[7, 2, 5], [0, 8, 3]], dtype=np.int32)
    lens = np.array([7, 10], dtype=np.int32)      # histories after the append
    n_new = 3
    lat, rope = _rows(rng, 2 * n_new)
    out = oracle.kv_append(slab, table, lens, lat, rope, n_new, page_tokens=page_tokens,
                           dc=DC, dr=DR)
    expect = slab.copy().reshape(-1)
    for r in range(2):
        for j in range(n_new):
            p = lens[r] - n_new + j                # positions 4..6 and 7..9: both cross a page
            base = table[r, p // page_tokens] * page_tokens * ROW + (p % page_tokens) * ROW
            expect[base:base + DC] = lat[r * n_new + j]
            expect[base + DC:base + ROW] = rope[r * n_new + j]
    assert np.array_equal(out.reshape(-1), expect)
    changed = np.nonzero(out.reshape(-1) != slab.reshape(-1))[0]
    assert changed.size <= 2 * n_new * ROW        # only the appended rows


def test_token_by_token_equals_one_append_of_the_history():
    rng = np.random.Generator(np.random.PCG64(2))
    page_tokens, num_pages = 4, 6
    slab0 = np.zeros((num_pages, page_tokens * ROW), dtype=np.uint16)
    table = np.array([[4, 1, 5, 0]], dtype=np.int32)
    L = 13
    lat, rope = _rows(rng, L)
    whole = oracle.kv_append(slab0, table, [L], lat, rope, L, page_tokens=page_tokens,
                             dc=DC, dr=DR)
    step = slab0
    for t in range(L):
        step = oracle.kv_append(step, table, [t + 1], lat[t:t + 1], rope[t:t + 1], 1,
                                page_tokens=page_tokens, dc=DC, dr=DR)
    assert np.array_equal(whole, step)


def test_decode_after_append_is_the_softmax_over_the_explicit_rows():
    rng = np.random.Generator(np.random.PCG64(3))
    page_tokens, num_pages, H = 4, 12, 2
    old_len, n_new = 6, 3
    table = np.array([[9, 3, 6], [1, 10, 0]], dtype=np.int32)
    hist_lat, hist_rope = _rows(rng, 2 * old_len)
    slab = np.zeros((num_pages, page_tokens * ROW), dtype=np.uint16)
    slab = oracle.kv_append(slab, table, [old_len, old_len], hist_lat, hist_rope, old_len,
                            page_tokens=page_tokens, dc=DC, dr=DR)
    new_lat, new_rope = _rows(rng, 2 * n_new)
    L = old_len + n_new
    slab = oracle.kv_append(slab, table, [L, L], new_lat, new_rope, n_new,
                            page_tokens=page_tokens, dc=DC, dr=DR)
    qn = _bf16_bits(rng.standard_normal((2, H, DC)))
    qr = _bf16_bits(rng.standard_normal((2, H, DR)))
    scale = 0.3
    o, lse = oracle.attend_rows(qn, qr, slab, table, [L, L], 1, H, scale, num_pages=num_pages,
                                page_tokens=page_tokens, dc=DC, dr=DR, threads=1)
    for r in range(2):
        c = np.concatenate([_bits_to_f64(hist_lat[r * old_len:(r + 1) * old_len]),
                            _bits_to_f64(new_lat[r * n_new:(r + 1) * n_new])])
        k = np.concatenate([_bits_to_f64(hist_rope[r * old_len:(r + 1) * old_len]),
                            _bits_to_f64(new_rope[r * n_new:(r + 1) * n_new])])
        for h in range(H):
            s = scale * (c @ _bits_to_f64(qn[r, h]) + k @ _bits_to_f64(qr[r, h]))
            w = np.exp(s - s.max())
            row = r * H + h
            assert np.allclose(o[row], (w / w.sum()) @ c, rtol=1e-12, atol=1e-12)
            assert lse[row] == pytest.approx(s.max() + np.log(w.sum()), abs=1e-12)


def test_padded_page_stride_and_wide_table():
    rng = np.random.Generator(np.random.PCG64(4))
    page_tokens, num_pages, stride = 4, 5, 4 * ROW + 8
    slab = _bf16_bits(rng.standard_normal((num_pages, stride)))
    table = np.array([[3, 1, 4, 2, 0, 0, 0]], dtype=np.int32)   # only the first columns used
    lat, rope = _rows(rng, 2)
    out = oracle.kv_append(slab, table, [6], lat, rope, 2, page_tokens=page_tokens,
                           page_stride=stride, dc=DC, dr=DR)
    flat, ref = out.reshape(-1), slab.reshape(-1)
    for j, p in enumerate([4, 5]):
        base = table[0, p // page_tokens] * stride + (p % page_tokens) * ROW
        assert np.array_equal(flat[base:base + DC], lat[j])
        assert np.array_equal(flat[base + DC:base + ROW], rope[j])
    # the padding between pages never changes
    for page in range(num_pages):
        pad = slice(page * stride + page_tokens * ROW, (page + 1) * stride)
        assert np.array_equal(flat[pad], ref[pad])


def test_out_of_range_positions_and_pages_raise():
    slab = np.zeros((3, 4 * ROW), dtype=np.uint16)
    lat, rope = np.zeros((2, DC), np.uint16), np.zeros((2, DR), np.uint16)
    with pytest.raises(IndexError):   # two new tokens but a history of one
        oracle.kv_append(slab, [[0]], [1], lat, rope, 2, page_tokens=4, dc=DC, dr=DR)
    with pytest.raises(IndexError):   # page 3 of a 3-page pool
        oracle.kv_append(slab, [[3]], [2], lat, rope, 2, page_tokens=4, dc=DC, dr=DR)
