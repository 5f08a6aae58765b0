"""GPU parity of the KV append (through the C ABI) against the oracle: bit-exact
pools after the write, skipped rows for bad positions and pages (status word,
nothing written elsewhere), and a decode of histories built only by the append."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_parity, gpu_decode, oracle_decode, to_device
from paged_latent_attention_gb300 import api, inputs

pytestmark = pytest.mark.gpu

ROW = inputs.ROW_ELEMS
PT = inputs.PAGE_TOKENS


def _rand_bf16(rng, shape):
    return torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16)


def _bits(t):
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _append(slab_dev, table_np, lens_np, lat, rope, n_new, status=None):
    table = torch.as_tensor(np.ascontiguousarray(table_np), dtype=torch.int32, device="cuda")
    lens = torch.as_tensor(np.asarray(lens_np, dtype=np.int32), device="cuda")
    api.mla_kv_append(lat.cuda(), rope.cuda(), slab_dev, table, lens, n_new, status=status)


@pytest.mark.parametrize("lengths,n_new,table_ld,pad", [
    ([1000, 2000, 3100], 1, None, 0),
    ([1536, 1537, 3072], 4, None, 0),      # the new rows cross page boundaries
    ([5, 1536 * 2 + 3, 700], 3, 9, 0),     # a table wider than the pages used
    ([4000, 10, 1600], 2, None, 24),       # padding between pages
    ([3000] * 37, 2, None, 0),             # more rows than one CTA's eight warps
])
def test_append_matches_oracle_bit_exact(lengths, n_new, table_ld, pad):
    w = inputs.custom_workload(lengths, 1, 16, seed=3, spare_pages=2, table_ld=table_ld,
                               page_stride=PT * ROW + pad)
    slab = inputs.make_slab(w, "cpu", poison_nan=True)
    rng = np.random.Generator(np.random.PCG64(1))
    lat = _rand_bf16(rng, (w.num_reqs * n_new, 512))
    rope = _rand_bf16(rng, (w.num_reqs * n_new, 64))
    dev = slab.cuda()
    _append(dev, w.page_table, w.seq_lens, lat, rope, n_new)
    torch.cuda.synchronize()
    ref = oracle.kv_append(slab, w.page_table, w.seq_lens, lat, rope, n_new,
                           page_tokens=PT, page_stride=w.page_stride)
    assert np.array_equal(_bits(dev), ref)


def test_zero_new_tokens_writes_nothing():
    w = inputs.custom_workload([700], 1, 16, seed=5)
    slab = inputs.make_slab(w, "cuda")
    before = slab.clone()
    empty = torch.empty(0, 512, dtype=torch.bfloat16, device="cuda")
    api.mla_kv_append(empty, empty[:, :64].contiguous(), slab,
                      torch.as_tensor(w.page_table, device="cuda"),
                      torch.as_tensor(w.seq_lens, device="cuda"), 0)
    torch.cuda.synchronize()
    assert torch.equal(slab.view(torch.int16), before.view(torch.int16))


def test_bad_rows_are_skipped_and_reported():
    w = inputs.custom_workload([3000, 2000], 1, 16, seed=4, spare_pages=2)
    slab = inputs.make_slab(w, "cpu", poison_nan=True)
    rng = np.random.Generator(np.random.PCG64(2))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    # request 1's history (1) is shorter than its 2 new tokens: position -1 is
    # skipped, its token 1 still lands at position 0
    lens = np.array([3000, 1], dtype=np.int32)
    lat, rope = _rand_bf16(rng, (4, 512)), _rand_bf16(rng, (4, 64))
    dev = slab.cuda()
    _append(dev, w.page_table, lens, lat, rope, 2, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 32
    ref = oracle.kv_append(slab, w.page_table[:1], lens[:1], lat[:2], rope[:2], 2,
                           page_tokens=PT, page_stride=w.page_stride)
    ref = oracle.kv_append(ref, w.page_table[1:], [1], lat[3:], rope[3:], 1,
                           page_tokens=PT, page_stride=w.page_stride)
    assert np.array_equal(_bits(dev), ref)

    # a page ID outside the pool: that request's row is skipped, the other written
    table = w.page_table.copy()
    table[0, 2999 // PT] = w.num_pages + 5
    lat, rope = _rand_bf16(rng, (2, 512)), _rand_bf16(rng, (2, 64))
    status.zero_()
    dev = slab.cuda()
    _append(dev, table, w.seq_lens, lat, rope, 1, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 33
    ref = oracle.kv_append(slab, table[1:], w.seq_lens[1:], lat[1:], rope[1:], 1,
                           page_tokens=PT, page_stride=w.page_stride)
    assert np.array_equal(_bits(dev), ref)

    # a history longer than the table's row: the column past it is never read
    narrow = np.ascontiguousarray(w.page_table[:, :2])
    lens = np.array([2 * PT + 1, 2000], dtype=np.int32)
    status.zero_()
    dev = slab.cuda()
    _append(dev, narrow, lens, lat, rope, 1, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 33
    ref = oracle.kv_append(slab, narrow[1:], lens[1:], lat[1:], rope[1:], 1,
                           page_tokens=PT, page_stride=w.page_stride)
    assert np.array_equal(_bits(dev), ref)


def test_decode_of_histories_written_by_the_append():
    """Start from an all-NaN pool, write each history with the GPU append (one
    long prefix per request, then shared steps of 1 to 4 tokens that cross page
    boundaries), check the pool bit for bit against the oracle's appends, then
    decode it with four draft tokens against the oracle."""
    target = np.array([1400, 1700, 333], dtype=np.int32)
    w = inputs.custom_workload(target, 4, 16, seed=6, spare_pages=2)
    qn, qr, gate = inputs.make_queries(w, "cpu")
    rng = np.random.Generator(np.random.PCG64(7))
    R = w.num_reqs
    steps = [int(x) for x in rng.integers(1, 5, size=40)]
    start = target - sum(steps)
    slab = torch.full((w.num_pages, w.page_stride), float("nan"), dtype=torch.bfloat16,
                      device="cuda")
    ref = np.full((w.num_pages, w.page_stride), 0x7FC0, dtype=np.uint16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for r in range(R):                      # the prefix, one request per call
        n = int(start[r])
        lat, rope = _rand_bf16(rng, (n, 512)), _rand_bf16(rng, (n, 64))
        _append(slab, w.page_table[r:r + 1], [n], lat, rope, n, status)
        ref = oracle.kv_append(ref, w.page_table[r:r + 1], [n], lat, rope, n,
                               page_tokens=PT, page_stride=w.page_stride)
    cur = start.copy()
    for n in steps:                         # decode-style steps, all requests at once
        cur = cur + n
        lat, rope = _rand_bf16(rng, (R * n, 512)), _rand_bf16(rng, (R * n, 64))
        _append(slab, w.page_table, cur, lat, rope, n, status)
        ref = oracle.kv_append(ref, w.page_table, cur, lat, rope, n,
                               page_tokens=PT, page_stride=w.page_stride)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(cur, target)
    assert np.array_equal(_bits(slab), ref)
    d = to_device(w, qn, qr, gate, slab)
    out, lse = gpu_decode(w, d)
    ref_slab = torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16)
    ref_out, ref_lse = oracle_decode(w, qn, qr, gate, ref_slab)
    assert_parity(out, lse, ref_out, ref_lse, what="append then decode")
