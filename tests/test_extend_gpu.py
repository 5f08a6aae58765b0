"""GPU parity of a chunked extend (prefill over the pages): a chunk of new tokens
per request, causal among themselves, attending over the paged history that
already holds their rows.  Same bar as the decode: |out - ref| <= 1e-2 +
1e-2 |ref|, |lse - ref| <= 1e-3, on every row or on sampled rows."""
import numpy as np
import pytest
import torch

from helpers import (assert_parity, assert_parity_fp8, gpu_decode, gpu_decode_fp8, oracle_decode,
                     oracle_decode_fp8, sample_rows, to_device)
from paged_latent_attention_gb300 import inputs

pytestmark = pytest.mark.gpu


def _problem(lengths, n_q, H, seed, fp8=False):
    w = inputs.custom_workload(lengths, n_q, H, seed=seed, spare_pages=2)
    qn, qr, gate = inputs.make_queries(w, "cpu")
    slab = (inputs.make_slab_e4m3(w, "cpu", poison_nan=True) if fp8
            else inputs.make_slab(w, "cpu", poison_nan=True))
    return w, qn, qr, gate, slab


@pytest.mark.parametrize("lengths,n_q,H", [
    ([3000, 5200], 64, 64),        # 64 row groups per request
    ([256, 700, 1537], 256, 16),   # the largest chunk; the first request is all new tokens
    ([129, 4099], 37, 32),         # a chunk that is not a multiple of anything
])
def test_extend_matches_oracle(lengths, n_q, H):
    w, qn, qr, gate, slab = _problem(lengths, n_q, H, seed=40 + n_q)
    d = to_device(w, qn, qr, gate, slab)
    out, lse = gpu_decode(w, d)
    rows = sample_rows(w, heads_per_token=2, seed=3)
    ref_out, ref_lse = oracle_decode(w, qn, qr, gate, slab, rows=rows)
    assert_parity(out, lse, ref_out, ref_lse, rows=rows, what=f"extend n_q={n_q} H={H}")
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


def test_extend_first_tokens_see_only_their_prefix():
    """With the history equal to the chunk (a prefill from empty), token j sees
    j + 1 rows: check every head of the first, second and last token."""
    w, qn, qr, gate, slab = _problem([100], 100, 16, seed=44)
    d = to_device(w, qn, qr, gate, slab)
    out, lse = gpu_decode(w, d)
    rows = [t * 16 + h for t in (0, 1, 99) for h in range(16)]
    ref_out, ref_lse = oracle_decode(w, qn, qr, gate, slab, rows=rows)
    assert_parity(out, lse, ref_out, ref_lse, rows=rows, what="prefill from empty")


def test_extend_fp8_pages():
    w, qn, qr, gate, slab = _problem([2000, 4500], 64, 64, seed=45, fp8=True)
    d = to_device(w, qn, qr, gate, slab)
    kvs = inputs.KV_SCALE_E4M3
    out, lse = gpu_decode_fp8(w, d, kvs)
    rows = sample_rows(w, heads_per_token=2, seed=4)
    ref_out, ref_lse, bound = oracle_decode_fp8(w, qn, qr, gate, slab, kvs, rows=rows)
    assert_parity_fp8(out, lse, ref_out, ref_lse, bound, rows=rows, what="fp8 extend")


def test_extend_workload_sampled():
    w = inputs.make_workload("extend")
    qn, qr, gate = inputs.make_queries(w, "cuda")
    slab = inputs.make_slab(w, "cuda")
    d = dict(qn=qn, qr=qr, gate=gate, slab=slab,
             table=torch.as_tensor(w.page_table, device="cuda"),
             lens=torch.as_tensor(w.seq_lens, device="cuda"))
    out, lse = gpu_decode(w, d)
    rng = np.random.Generator(np.random.PCG64(5))
    toks = sorted({0, 1, w.n_q - 1} | set(int(x) for x in rng.integers(0, w.num_tokens, 12)))
    rows = [t * w.num_heads + h for t in toks for h in (0, 17, 63)]
    ref_out, ref_lse = oracle_decode(w, qn.cpu(), qr.cpu(), gate.cpu(), slab.cpu(), rows=rows)
    assert_parity(out, lse, ref_out, ref_lse, rows=rows, what="extend workload")
    assert torch.isfinite(lse).all() and torch.isfinite(out.float()).all()
