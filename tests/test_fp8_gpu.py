"""GPU parity of the FP8 (E4M3) page path against the oracle, through the C ABI.

Bar: query split (hi and lo codes, exponents) and FP8 append bytes bit-exact;
the decode against the pages' definition (the bf16 query over the dequantised
cache) within |lse - ref| <= 1e-3 + D and |out - ref| <= 1e-2 + 1e-2 |ref| +
((1 + 2^-4) e^{2D} - 1) A + 2^-14 e^{2D} B, the bound derived in helpers from
E4M3's arithmetic for the kernel's two-part query and E4M3 probabilities; page
indexing exact (one-hot probes).
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import (SCALE, assert_parity_fp8, gpu_decode_fp8, oracle_decode_fp8, sample_rows,
                     to_device)
from paged_latent_attention_gb300 import api, inputs

pytestmark = pytest.mark.gpu

PT = inputs.PAGE_TOKENS
ROW = inputs.ROW_ELEMS
KVS = inputs.KV_SCALE_E4M3


def _problem(lengths, n_q, H, seed, spare=3, page_pad=0, poison=True, kv_scale=KVS):
    w = inputs.custom_workload(lengths, n_q, H, seed=seed, spare_pages=spare,
                               page_stride=PT * ROW + page_pad)
    qn, qr, gate = inputs.make_queries(w, "cpu")
    slab = inputs.make_slab_e4m3(w, "cpu", poison_nan=poison, kv_scale=kv_scale)
    return w, qn, qr, gate, slab


def test_query_quantiser_is_bit_exact():
    g = torch.Generator().manual_seed(3)
    rows = 300
    qn = torch.randn(rows, 512, generator=g)
    qr = torch.randn(rows, 64, generator=g)
    mag = torch.tensor([10.0 ** k for k in np.linspace(-30, 30, rows)], dtype=torch.float32)
    qn, qr = (qn * mag[:, None]).bfloat16(), (qr * mag[:, None]).bfloat16()
    qn[7].zero_()
    qr[7].zero_()                                   # all-zero row: e = 0
    qn[8, 3] = 448.0                                # the row maximum exactly 448
    qr[9, 0] = -3.0e38                              # near bf16's largest finite
    hi, lo, exps = api.mla_quantize_queries_fp8(qn.cuda(), qr.cuda())
    ref_hi, ref_lo, ref_exps = oracle.quantize_query_rows(qn, qr)
    assert np.array_equal(exps.cpu().numpy(), ref_exps)
    assert np.array_equal(hi.cpu().numpy(), ref_hi)
    assert np.array_equal(lo.cpu().numpy(), ref_lo)


RAGGED = [1, 2, 127, 128, 129, 1535, 1536, 1537, 4099]


@pytest.mark.parametrize("n_q,H", [(1, 16), (1, 32), (1, 64), (4, 64), (3, 16), (1, 128)])
@pytest.mark.parametrize("cta_budget,min_splits", [(0, 1), (4, 1), (0, 9)])
def test_ragged_histories_fp8(n_q, H, cta_budget, min_splits):
    w, qn, qr, gate, slab = _problem(RAGGED, n_q, H, seed=300 + n_q * 7 + H)
    d = to_device(w, qn, qr, gate, slab)
    out, lse = gpu_decode_fp8(w, d, KVS, cta_budget=cta_budget, min_splits=min_splits)
    ref_out, ref_lse, bound = oracle_decode_fp8(w, qn, qr, gate, slab, KVS)
    assert_parity_fp8(out, lse, ref_out, ref_lse, bound, what=f"fp8 ragged n_q={n_q} H={H}")


@pytest.mark.parametrize("kv_scale", [1.0 / 64, 0.0371, 3.0])
def test_kv_scales_and_padded_stride(kv_scale):
    w, qn, qr, gate, slab = _problem([1600, 4000, 300], 1, 64, seed=31, page_pad=48,
                                     kv_scale=kv_scale)
    d = to_device(w, qn, qr, gate, slab)
    out, lse = gpu_decode_fp8(w, d, kv_scale)
    ref_out, ref_lse, bound = oracle_decode_fp8(w, qn, qr, gate, slab, kv_scale)
    assert_parity_fp8(out, lse, ref_out, ref_lse, bound, what=f"kv_scale={kv_scale}")


def test_empty_history_fp8():
    w, qn, qr, gate, slab = _problem([0, 300, 0], 1, 16, seed=32)
    w.page_table[0, :] = w.page_table[1, 0]
    d = to_device(w, qn, qr, gate, slab)
    out, lse = gpu_decode_fp8(w, d, KVS)
    o = out.float().cpu().view(3, 16, 512)
    l = lse.cpu().view(3, 16)
    assert torch.all(o[0] == 0) and torch.all(o[2] == 0)
    assert torch.all(torch.isneginf(l[0])) and torch.all(torch.isneginf(l[2]))


def test_one_hot_probe_fp8_pages():
    """q_rope = 2^10 e_5 (an exact E4M3 code after the query scale), one token
    whose rope byte 5 decodes to 1 / kv_scale, gate +100: the probability of
    that token is 2^4 exactly in E4M3, every other one underflows to 0, so the
    output is the token's dequantised latent row to bf16 rounding."""
    kv_scale = 1.0 / 16
    L = 3 * PT + 17
    w, qn, qr, gate, slab = _problem([L, 700], 1, 16, seed=33, spare=3, kv_scale=kv_scale)
    pages = slab.view(w.num_pages, PT, ROW)
    pages[..., 512:] = 0
    qn.zero_()
    qr.zero_()
    qr[:, :, 5] = 2.0 ** 10
    gate.fill_(100.0)
    one = int(oracle.e4m3_encode([16.0])[0])        # decodes to 16: value 16 * kv_scale = 1
    d = to_device(w, qn, qr, gate, slab)
    dev_pages = d["slab"].view(w.num_pages, PT, ROW)
    for t_star in [0, 1, PT - 1, PT, 2 * PT - 1, 2 * PT, 3 * PT - 1, 3 * PT, L - 1]:
        p = int(w.page_table[0, t_star // PT])
        dev_pages[..., 512 + 5] = 0
        dev_pages[p, t_star % PT, 512 + 5] = one
        for budget, min_splits in [(0, 1), (0, 16)]:
            out, lse = gpu_decode_fp8(w, d, kv_scale, cta_budget=budget, min_splits=min_splits)
            row = dev_pages[p, t_star % PT, :512].cpu().numpy()
            expect = torch.from_numpy(kv_scale * oracle.e4m3_decode(row)).to(torch.bfloat16)
            assert torch.equal(out[0].view(16, 512).cpu(), expect.expand(16, 512)), t_star
            assert torch.allclose(lse[0].cpu(), torch.full((16,), SCALE * 2.0 ** 10), atol=1e-3)


def test_page_permutation_is_bit_identical_fp8():
    w, qn, qr, gate, slab = _problem([5000, 1537, 9000], 1, 64, seed=34, spare=6)
    d = to_device(w, qn, qr, gate, slab)
    out1, lse1 = gpu_decode_fp8(w, d, KVS)
    out2, lse2 = gpu_decode_fp8(w, d, KVS)
    perm = np.random.Generator(np.random.PCG64(1)).permutation(w.num_pages)
    inv = np.argsort(perm)
    d["slab"] = d["slab"][torch.as_tensor(perm, device="cuda")].contiguous()
    d["table"] = torch.as_tensor(inv[w.page_table].astype(np.int32), device="cuda")
    out3, lse3 = gpu_decode_fp8(w, d, KVS)
    for o, l in [(out2, lse2), (out3, lse3)]:
        assert torch.equal(out1.view(torch.int16), o.view(torch.int16))
        assert torch.equal(lse1, l)


@pytest.mark.parametrize("lengths,n_new,pad", [
    ([1000, 2000, 3100], 1, 0),
    ([1536, 1537, 3072], 4, 0),
    ([4000, 10, 1600], 2, 32),
])
def test_fp8_append_bit_exact(lengths, n_new, pad):
    w = inputs.custom_workload(lengths, 1, 16, seed=35, spare_pages=2, page_stride=PT * ROW + pad)
    slab = inputs.make_slab_e4m3(w, "cpu", poison_nan=True)
    g = torch.Generator().manual_seed(5)
    lat = (torch.randn(w.num_reqs * n_new, 512, generator=g) * 3).bfloat16()
    rope = torch.randn(w.num_reqs * n_new, 64, generator=g).bfloat16()
    lat[0, :4] = torch.tensor([1e6, -1e6, 0.0, -0.0])      # saturation and signed zeros
    dev = slab.cuda()
    api.mla_kv_append_fp8(lat.cuda(), rope.cuda(), dev, torch.as_tensor(w.page_table, device="cuda"),
                          torch.as_tensor(w.seq_lens, device="cuda"), n_new, kv_scale=KVS)
    torch.cuda.synchronize()
    ref = oracle.kv_append_e4m3(slab, w.page_table, w.seq_lens, lat, rope, n_new, KVS,
                                page_stride=w.page_stride)
    assert np.array_equal(dev.cpu().numpy(), ref)


def test_fp8_append_then_decode():
    target = np.array([1400, 1700, 333], dtype=np.int32)
    w = inputs.custom_workload(target, 4, 64, seed=36, spare_pages=2)
    qn, qr, gate = inputs.make_queries(w, "cpu")
    slab = torch.full((w.num_pages, w.page_stride), inputs.E4M3_NAN, dtype=torch.uint8,
                      device="cuda")
    ref = np.full((w.num_pages, w.page_stride), inputs.E4M3_NAN, dtype=np.uint8)
    g = torch.Generator().manual_seed(6)
    for r in range(w.num_reqs):
        n = int(target[r])
        lat, rope = torch.randn(n, 512, generator=g).bfloat16(), torch.randn(n, 64, generator=g).bfloat16()
        api.mla_kv_append_fp8(lat.cuda(), rope.cuda(), slab,
                              torch.as_tensor(w.page_table[r:r + 1], device="cuda"),
                              torch.as_tensor([n], dtype=torch.int32, device="cuda"), n,
                              kv_scale=KVS)
        ref = oracle.kv_append_e4m3(ref, w.page_table[r:r + 1], [n], lat, rope, n, KVS)
    torch.cuda.synchronize()
    assert np.array_equal(slab.cpu().numpy(), ref)
    d = to_device(w, qn, qr, gate, slab)
    out, lse = gpu_decode_fp8(w, d, KVS)
    ref_out, ref_lse, bound = oracle_decode_fp8(w, qn, qr, gate, ref, KVS)
    assert_parity_fp8(out, lse, ref_out, ref_lse, bound, what="fp8 append then decode")


@pytest.mark.parametrize("name,heads", [("steady", 4), ("spec", 1)])
def test_fp8_workload_parity_sampled(name, heads):
    w = inputs.make_workload(name)
    qn, qr, gate = inputs.make_queries(w, "cuda")
    slab = inputs.make_slab_e4m3(w, "cuda")
    d = dict(qn=qn, qr=qr, gate=gate, slab=slab,
             table=torch.as_tensor(w.page_table, device="cuda"),
             lens=torch.as_tensor(w.seq_lens, device="cuda"))
    out, lse = gpu_decode_fp8(w, d, KVS)
    rows = sample_rows(w, heads_per_token=heads, seed=2)
    host = slab.cpu()
    ref_out, ref_lse, bound = oracle_decode_fp8(w, qn.cpu(), qr.cpu(), gate.cpu(), host, KVS,
                                                rows=rows)
    assert_parity_fp8(out, lse, ref_out, ref_lse, bound, rows=rows, what=f"fp8 {name}")
    assert torch.isfinite(lse).all() and torch.isfinite(out.float()).all()
