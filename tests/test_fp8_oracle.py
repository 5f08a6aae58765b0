"""Pins for the oracle's FP8 (E4M3) pages, FP8 queries and FP8 KV append (CPU only).

The codec is checked against torch's float8_e4m3fn (a library implementation of
the same OCP format); FP8 attention is tied to the already pinned bf16 oracle by
building bf16 pages that hold exactly the dequantised values; the query
quantisation against its definition (smallest power-of-two scale that keeps the
row inside E4M3's range) by brute force.
"""
import numpy as np
import pytest
import torch

import oracle

DC, DR = 8, 4
ROW = DC + DR


def _bf16_bits(x):
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _f64_to_bf16_exact(v):
    """bf16 bits of values that bf16 represents exactly (asserted)."""
    b = _bf16_bits(v)
    back = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(back, np.asarray(v, dtype=np.float64))
    return b


def _torch_e4m3(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def test_decode_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.array_equal(ours[~np.isnan(ours)], ref[~np.isnan(ref)])
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_encode_matches_torch_in_range_and_rounds_ties_to_even():
    rng = np.random.Generator(np.random.PCG64(0))
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0)])
    x = x[np.abs(x) <= 448].astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(x), _torch_e4m3(x))
    # every representable value round-trips
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(finite)), finite)
    # exact midpoints between neighbours go to the even code
    tab = oracle.e4m3_decode(np.arange(127, dtype=np.uint8))
    mids = (tab[:-1] + tab[1:]) / 2
    codes = oracle.e4m3_encode(mids)
    assert np.all(codes % 2 == 0)
    assert np.all((codes == np.arange(126)) | (codes == np.arange(1, 127)))
    assert np.array_equal(codes, _torch_e4m3(mids.astype(np.float32)))


def test_encode_saturates_keeps_sign_and_maps_nan():
    assert oracle.e4m3_encode([1000.0, -1e30, 464.0, 449.0]).tolist() == [0x7E, 0xFE, 0x7E, 0x7E]
    assert oracle.e4m3_encode([-0.0, 0.0, -1e-6]).tolist() == [0x80, 0x00, 0x80]
    assert oracle.e4m3_encode([np.nan]).tolist() == [0x7F]


def test_query_scale_is_the_smallest_power_of_two_that_fits():
    rng = np.random.Generator(np.random.PCG64(1))
    amax = np.concatenate([np.abs(rng.standard_normal(500)) * 10.0 ** rng.integers(-6, 6, 500),
                           [448.0, 448.0 * 2 ** 5, 1.75, 1.7500001, 2.0 ** -20, 1.0]])
    e = oracle.query_scale_exponent(amax)
    for a, k in zip(amax, e):
        assert a * 2.0 ** -int(k) <= 448.0
        assert a * 2.0 ** -(int(k) - 1) > 448.0       # one power smaller would not fit
    assert oracle.query_scale_exponent([0.0]).tolist() == [0]
    assert oracle.query_scale_exponent([448.0]).tolist() == [0]


def test_two_part_query_is_exact_above_a_quarter_of_the_scale():
    """The split the FP8 decode's tolerance relies on, by brute force over every
    finite bf16 magnitude up to the row maximum: (hi + lo) * 2^e equals q
    exactly where |q| >= 2^(e - 2), and is within 2^(e - 10) below that; hi
    alone is within 2^-4 relative in E4M3's normal range."""
    mags = np.arange(0, 0x43E1, dtype=np.uint16)          # +0 .. 448 as bf16 bit patterns
    vals = oracle.oracle._bf16_to_f64(mags)
    assert vals.max() == 448.0
    for scale_exp in (0, -7, 5):
        q = np.concatenate([vals, -vals]) * 2.0 ** scale_exp
        pad = (-q.size) % ROW
        q = np.concatenate([q, np.zeros(pad)]).reshape(-1, ROW)
        q[:, 0] = 400.0 * 2.0 ** scale_exp                # every row's maximum: e = scale_exp
        qn = _bf16_bits(q[:, :DC])
        qr = _bf16_bits(q[:, DC:])
        hi, lo, e = oracle.quantize_query_rows(qn, qr)
        assert np.all(e == scale_exp)
        back = oracle.dequantize_query_rows(hi, lo, e)
        big = np.abs(q) >= 2.0 ** (scale_exp - 2)
        assert np.array_equal(back[big], q[big])
        assert np.abs(back - q)[~big].max() <= 2.0 ** (scale_exp - 10)
        hi_only = np.ldexp(oracle.e4m3_decode(hi), e[:, None].astype(np.int64))
        normal = np.abs(q) >= 2.0 ** (scale_exp - 6)
        assert (np.abs(hi_only - q)[normal] / np.abs(q)[normal]).max() <= 2.0 ** -4


def test_query_scale_puts_the_row_maximum_in_the_top_binade():
    rng = np.random.Generator(np.random.PCG64(2))
    qn = _bf16_bits(rng.standard_normal((6, DC)) * np.array([1, 1e-3, 100, 5, 1, 0.01])[:, None])
    qr = _bf16_bits(rng.standard_normal((6, DR)))
    hi, lo, e = oracle.quantize_query_rows(qn, qr)
    assert hi.shape == (6, ROW) and lo.shape == (6, ROW) and hi.dtype == np.uint8
    q = np.concatenate([oracle.oracle._bf16_to_f64(qn), oracle.oracle._bf16_to_f64(qr)], axis=1)
    amax = np.abs(q).max(axis=1)
    assert np.all(amax * 2.0 ** -e > 224.0) and np.all(amax * 2.0 ** -e <= 448.0)


def _random_fp8_pool(rng, num_pages, page_tokens):
    codes = rng.integers(0, 256, size=(num_pages, page_tokens * ROW)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C          # no NaN codes inside a history
    return codes


@pytest.mark.parametrize("kv_scale", [0.125, 1.0, 4.0])
def test_fp8_attention_equals_bf16_oracle_on_the_dequantised_pool(kv_scale):
    """With a power-of-two kv_scale, kv_scale * decoded byte is a bf16 value, so
    attention over the FP8 pool must equal the pinned bf16 oracle over a bf16
    pool holding those values, bit for bit (identical double arithmetic)."""
    rng = np.random.Generator(np.random.PCG64(3))
    pt, pages, H, n_q = 4, 10, 2, 2
    pool8 = _random_fp8_pool(rng, pages, pt)
    pool16 = _f64_to_bf16_exact(kv_scale * oracle.e4m3_decode(pool8))
    table = np.array([[7, 1, 4], [0, 9, 5]], dtype=np.int32)
    lens = np.array([11, 7], dtype=np.int32)
    qn = _bf16_bits(rng.standard_normal((2 * n_q, H, DC)))
    qr = _bf16_bits(rng.standard_normal((2 * n_q, H, DR)))
    a = oracle.attend_rows(qn, qr, pool8, table, lens, n_q, H, 0.2, num_pages=pages,
                           page_tokens=pt, dc=DC, dr=DR, kv_format="e4m3", kv_scale=kv_scale)
    b = oracle.attend_rows(qn, qr, pool16, table, lens, n_q, H, 0.2, num_pages=pages,
                           page_tokens=pt, dc=DC, dr=DR)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_fp8_kv_scale_factors_out_of_scores_and_outputs():
    rng = np.random.Generator(np.random.PCG64(4))
    pt, pages, H = 4, 6, 3
    pool8 = _random_fp8_pool(rng, pages, pt)
    table = np.array([[2, 5, 0]], dtype=np.int32)
    lens = np.array([10], dtype=np.int32)
    qn = _bf16_bits(rng.standard_normal((1, H, DC)))
    qr = _bf16_bits(rng.standard_normal((1, H, DR)))
    c = 0.37
    o1, l1 = oracle.attend_rows(qn, qr, pool8, table, lens, 1, H, 0.1, num_pages=pages,
                                page_tokens=pt, dc=DC, dr=DR, kv_format="e4m3", kv_scale=c)
    o2, l2 = oracle.attend_rows(qn, qr, pool8, table, lens, 1, H, 0.1 * c, num_pages=pages,
                                page_tokens=pt, dc=DC, dr=DR, kv_format="e4m3", kv_scale=1.0)
    assert np.allclose(o1, c * o2, rtol=1e-12, atol=1e-14)
    assert np.allclose(l1, l2, rtol=0, atol=1e-12)


def test_fp8_decode_is_the_softmax_over_explicit_dequantised_rows():
    """The E4M3 reference is the bf16 query over the dequantised rows, and its
    bound terms are what they claim: A = sigmoid(g) sum_t w_t |c_t|,
    B = sigmoid(g) w_max sum_t |c_t|, D = max_t |scale| sum_d eps_d |x_t,d|."""
    rng = np.random.Generator(np.random.PCG64(5))
    pt, pages, H, n_q = 4, 8, 2, 1
    pool8 = _random_fp8_pool(rng, pages, pt)
    table = np.array([[3, 6], [1, 0]], dtype=np.int32)
    lens = np.array([7, 5], dtype=np.int32)
    qn = _bf16_bits(rng.standard_normal((2, H, DC)) * 3)
    qr = _bf16_bits(rng.standard_normal((2, H, DR)))
    gate = _bf16_bits(rng.standard_normal((2, H, DC)))
    eps = rng.random((2 * H, ROW)) * (rng.random((2 * H, ROW)) < 0.1)
    kv_scale, scale = 0.5, -0.25
    out, lse, terms = oracle.mla_decode_e4m3_reference(
        qn, qr, gate, pool8, kv_scale, table, lens, n_q, H, scale, num_pages=pages,
        page_tokens=pt, dc=DC, dr=DR, with_abs=True, query_err=eps)
    q = np.concatenate([oracle.oracle._bf16_to_f64(qn).reshape(-1, DC),
                        oracle.oracle._bf16_to_f64(qr).reshape(-1, DR)], axis=1)
    g = oracle.oracle._bf16_to_f64(gate).reshape(-1, DC)
    for r in range(2):
        rows = [pool8[table[r, t // pt], (t % pt) * ROW:(t % pt + 1) * ROW] for t in range(lens[r])]
        x = kv_scale * oracle.e4m3_decode(np.stack(rows))
        for h in range(H):
            i = r * H + h
            s = scale * (x @ q[i])
            w = np.exp(s - s.max())
            w /= w.sum()
            sig = 1.0 / (1.0 + np.exp(-g[i]))
            assert np.allclose(out[i], sig * (w @ x[:, :DC]), rtol=1e-12, atol=1e-14)
            assert np.allclose(terms["A"][i], sig * (w @ np.abs(x[:, :DC])), rtol=1e-12,
                               atol=1e-14)
            assert np.allclose(terms["B"][i], sig * w.max() * np.abs(x[:, :DC]).sum(axis=0),
                               rtol=1e-12, atol=1e-14)
            assert terms["D"][i] == pytest.approx(abs(scale) * (np.abs(x) @ eps[i]).max(),
                                                  rel=1e-12)
            assert lse[i] == pytest.approx(s.max() + np.log(np.exp(s - s.max()).sum()), abs=1e-12)


def test_derived_fp8_bound_covers_the_two_part_query_and_e4m3_probabilities():
    """The tolerance the GPU tests use (tests/helpers.py), checked against a
    double-precision model of the two documented approximations on a random
    problem: the two-part query (exact dequantised values) and E4M3-rounded
    probabilities 2^(x - m + 4) with fp32 normaliser.  A plausible mistake in the
    bound (dropping a term, the wrong sign of D) fails here first."""
    import helpers
    rng = np.random.Generator(np.random.PCG64(9))
    pt, pages, H = 8, 40, 4
    pool8 = _random_fp8_pool(rng, pages, pt)
    pool8[rng.random(pool8.shape) < 0.5] = 0x30         # a skewed pool: sharper softmax
    lens = np.array([300, 17, 1], dtype=np.int32)
    table = np.stack([rng.permutation(pages)[:38] for _ in range(3)]).astype(np.int32)
    qn = _bf16_bits(rng.standard_normal((3, H, DC)) * 4)
    qr = _bf16_bits(rng.standard_normal((3, H, DR)))
    qn[0, 0, :4] = _bf16_bits(rng.standard_normal(4) * 1e-4)   # elements below 2^(e-2)
    gate = _bf16_bits(rng.standard_normal((3, H, DC)))
    kvs, scale = 0.05, 0.072
    eps = helpers.fp8_query_error(qn, qr)
    ref, ref_lse, terms = oracle.mla_decode_e4m3_reference(
        qn, qr, gate, pool8, kvs, table, lens, 1, H, scale, num_pages=pages, page_tokens=pt,
        dc=DC, dr=DR, with_abs=True, query_err=eps)
    hi, lo, e = oracle.quantize_query_rows(qn, qr)
    qd = oracle.dequantize_query_rows(hi, lo, e)
    tol, ltol = helpers.fp8_tolerance(ref, terms)
    g = oracle.oracle._bf16_to_f64(gate).reshape(-1, DC)
    for r in range(3):
        x = kvs * oracle.e4m3_decode(np.stack(
            [pool8[table[r, t // pt], (t % pt) * ROW:(t % pt + 1) * ROW] for t in range(lens[r])]))
        for h in range(H):
            i = r * H + h
            s = scale * (x @ qd[i]) * np.log2(np.e)          # the kernel's scores, log2 units
            p = np.exp2(s - s.max() + 4.0)
            p8 = oracle.e4m3_decode(oracle.e4m3_encode(p))
            o = (p8 @ x[:, :DC]) / p.sum()
            out = o / (1.0 + np.exp(-g[i]))
            lse = (s.max() - 4.0 + np.log2(p.sum())) * np.log(2.0)
            assert np.all(np.abs(out - ref[i]) <= tol[i] - 1e-2)   # inside the derived part alone
            assert abs(lse - ref_lse[i]) <= ltol[i]
    assert terms["D"][0] > 0.0


def test_derived_fp8_bound_needs_each_of_its_terms():
    """Two constructed rows where the model's error comes close to one term of
    the bound, so that dropping that term (or flipping the sign of D) fails.
    Head 0: one token at the maximum and 10,000 equal tokens 13.51 log2 units
    below it, whose probabilities 0.7 * 2^-9 all round up to the subnormal step
    2^-9 (the B term).  Head 1: eleven query elements of 0.6 * 2^-17 whose lo
    parts all round the same way, shifting every score by 0.8 D (the D term)."""
    import helpers
    pt, n = 8, 10_001
    pages = -(-n // pt)
    row = np.full(ROW, 0x7E, dtype=np.uint8)          # 448 everywhere but element 0
    row[0] = 0x00
    pool8 = np.tile(row, (pages, pt))
    pool8[0, 0] = 0x38                                # token 0: element 0 = 1.0
    table = np.arange(pages, dtype=np.int32)[None, :]
    lens = np.array([n], dtype=np.int32)
    q = np.zeros((1, 2, ROW))
    q[0, :, 0] = 1.0
    q[0, 1, 1:] = 0.6 * 2.0 ** -17
    qn, qr = _bf16_bits(q[..., :DC]), _bf16_bits(q[..., DC:])
    gate = _bf16_bits(np.zeros((1, 2, DC)))
    scale = (13.0 - np.log2(0.7) + 4.0 - 4.0) / np.log2(np.e)   # 13.51 log2 units per unit
    eps = helpers.fp8_query_error(qn, qr)
    ref, ref_lse, terms = oracle.mla_decode_e4m3_reference(
        qn, qr, gate, pool8, 1.0, table, lens, 1, 2, scale, num_pages=pages, page_tokens=pt,
        dc=DC, dr=DR, with_abs=True, query_err=eps)
    hi, lo, e = oracle.quantize_query_rows(qn, qr)
    qd = oracle.dequantize_query_rows(hi, lo, e)
    x = oracle.e4m3_decode(pool8.reshape(-1, ROW)[:n])
    assert terms["D"][0] == 0.0 and terms["D"][1] > 0.1
    tol, ltol = helpers.fp8_tolerance(ref, terms)
    for h in range(2):
        s = scale * (x @ qd[h]) * np.log2(np.e)
        p = np.exp2(s - s.max() + 4.0)
        p8 = oracle.e4m3_decode(oracle.e4m3_encode(p))
        out = 0.5 * (p8 @ x[:, :DC]) / p.sum()
        lse = (s.max() - 4.0 + np.log2(p.sum())) * np.log(2.0)
        err = np.abs(out - ref[h])
        assert np.all(err <= tol[h] - 1e-2 - 1e-2 * np.abs(ref[h]))
        assert abs(lse - ref_lse[h]) <= ltol[h]
        if h == 0:       # the B term carries it: the rest of the bound is too small
            rest = ((1 + helpers.P_E4M3_REL) * np.exp(2 * terms["D"][0]) - 1) * terms["A"][0]
            assert err[1:].max() > 2 * rest[1:].max()
        else:            # the LSE moves by most of D
            assert abs(lse - ref_lse[h]) > 0.5 * terms["D"][1] > 1e-2


def test_fp8_append_lands_rows_as_codes_of_the_scaled_values():
    rng = np.random.Generator(np.random.PCG64(6))
    pt, pages = 4, 7
    slab = _random_fp8_pool(rng, pages, pt)
    table = np.array([[6, 2, 3], [1, 4, 0]], dtype=np.int32)
    lens = np.array([6, 9], dtype=np.int32)
    n_new, kv_scale = 3, 0.3
    lat = _bf16_bits(rng.standard_normal((2 * n_new, DC)) * 20)
    rope = _bf16_bits(rng.standard_normal((2 * n_new, DR)))
    out = oracle.kv_append_e4m3(slab, table, lens, lat, rope, n_new, kv_scale, page_tokens=pt,
                                dc=DC, dr=DR)
    expect = slab.copy().reshape(-1)
    lat32 = oracle.oracle._bf16_to_f64(lat).astype(np.float32)
    rope32 = oracle.oracle._bf16_to_f64(rope).astype(np.float32)
    for r in range(2):
        for j in range(n_new):
            p = lens[r] - n_new + j
            base = table[r, p // pt] * pt * ROW + (p % pt) * ROW
            vals = np.concatenate([lat32[r * n_new + j], rope32[r * n_new + j]]) / np.float32(kv_scale)
            expect[base:base + ROW] = _torch_e4m3(vals)
    assert np.array_equal(out.reshape(-1), expect)
    # the stored rows decode to the inputs within half an FP8 step
    got = kv_scale * oracle.e4m3_decode(out.reshape(-1)[expect != slab.reshape(-1)])
    assert got.size > 0
    with pytest.raises(IndexError):
        oracle.kv_append_e4m3(slab, [[0]], [1], lat[:2], rope[:2], 2, 1.0, page_tokens=pt,
                              dc=DC, dr=DR)
