"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
(via the torch front end) and the double-precision oracle on the same inputs."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from paged_latent_attention_gb300 import api, inputs

SCALE = 1.0 / math.sqrt(192.0)
OUT_ATOL = 1e-2   # |out - ref| <= OUT_ATOL + OUT_RTOL * |ref|  (bf16 output)
OUT_RTOL = 1e-2
LSE_ATOL = 1e-3   # |lse - ref| <= LSE_ATOL                      (fp32 log-sum-exp)


def to_device(w: inputs.Workload, qn, qr, gate, slab, device="cuda"):
    return dict(
        qn=qn.to(device), qr=qr.to(device), gate=gate.to(device), slab=slab.to(device),
        table=torch.as_tensor(w.page_table, dtype=torch.int32, device=device),
        lens=torch.as_tensor(w.seq_lens, dtype=torch.int32, device=device))


def gpu_decode(w, d, *, cta_budget=0, min_splits=None, scale=SCALE):
    ms = min_splits or w.min_splits
    ws = api.allocate_workspace(w.num_reqs, w.n_q, w.num_heads, cta_budget, ms, "cuda")
    out, lse = api.mla_decode(d["qn"], d["qr"], d["gate"], d["slab"], d["table"], d["lens"],
                              n_q=w.n_q, scale=scale, cta_budget=cta_budget, min_splits=ms,
                              workspace=ws)
    torch.cuda.synchronize()
    assert api.device_status(ws) == 0, "a decode pipeline wait timed out"
    return out, lse


def oracle_decode(w, qn, qr, gate, slab_host, rows=None, scale=SCALE):
    return oracle.mla_decode_reference(qn, qr, gate, slab_host, w.page_table, w.seq_lens,
                                       w.n_q, w.num_heads, scale, num_pages=w.num_pages,
                                       page_stride=w.page_stride, page_tokens=w.page_tokens,
                                       dc=w.dc, dr=w.dr, rows=rows)


def assert_parity(out, lse, ref_out, ref_lse, rows=None, what=""):
    o = out.float().cpu().numpy().reshape(-1, out.shape[-1]).astype(np.float64)
    l = lse.cpu().numpy().reshape(-1).astype(np.float64)
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        o, l = o[rows], l[rows]
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    err = np.abs(o - ref_out)
    bound = OUT_ATOL + OUT_RTOL * np.abs(ref_out)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} outputs out of tolerance, "
                           f"max err {err.max():.3e}")
    both_inf = np.isneginf(l) & np.isneginf(ref_lse)
    with np.errstate(invalid="ignore"):
        lerr = np.where(both_inf, 0.0, np.abs(l - ref_lse))
    assert np.all(lerr <= LSE_ATOL), f"{what}: lse max err {np.nanmax(lerr):.3e}"
    return float(err.max()), float(lerr.max())


def sample_rows(w, heads_per_token=4, seed=0):
    """Every (request, draft) row set restricted to a few heads, incl. first and last."""
    rng = np.random.Generator(np.random.PCG64(seed))
    H = w.num_heads
    rows = []
    for t in range(w.num_tokens):
        hs = {0, H - 1}
        while len(hs) < min(H, heads_per_token):
            hs.add(int(rng.integers(0, H)))
        rows.extend(t * H + h for h in sorted(hs))
    return np.array(rows, dtype=np.int64)


# --------------------------------------------------------------------------
# FP8 (E4M3) pages
# --------------------------------------------------------------------------

# The FP8 decode rounds each probability to E4M3 before the value MMA (3
# mantissa bits: relative error <= 2^-4), while the normaliser and the LSE use
# the fp32 probabilities.  So |out - ref| may exceed the bf16 bound by at most
# 2^-4 * sigmoid(g) * sum_t w_t |c_t| (w = the exact softmax weights, c = the
# dequantised latent), which the oracle returns as `bound`.  The LSE bound is
# unchanged.
P_E4M3_REL = 2.0 ** -4


def gpu_decode_fp8(w, d, kv_scale, *, cta_budget=0, min_splits=None, scale=SCALE):
    ms = min_splits or w.min_splits
    ws = api.allocate_workspace(w.num_reqs, w.n_q, w.num_heads, cta_budget, ms, "cuda",
                                fp8=True)
    out, lse = api.mla_decode_fp8(d["qn"], d["qr"], d["gate"], d["slab"], d["table"], d["lens"],
                                  kv_scale=kv_scale, n_q=w.n_q, scale=scale,
                                  cta_budget=cta_budget, min_splits=ms, workspace=ws)
    torch.cuda.synchronize()
    assert api.device_status(ws) == 0, "a decode pipeline wait timed out"
    return out, lse


def oracle_decode_fp8(w, qn, qr, gate, slab8_host, kv_scale, rows=None, scale=SCALE):
    return oracle.mla_decode_e4m3_reference(qn, qr, gate, slab8_host, kv_scale, w.page_table,
                                            w.seq_lens, w.n_q, w.num_heads, scale,
                                            num_pages=w.num_pages, page_stride=w.page_stride,
                                            page_tokens=w.page_tokens, dc=w.dc, dr=w.dr,
                                            rows=rows, with_abs=True)


def assert_parity_fp8(out, lse, ref_out, ref_lse, bound, rows=None, what=""):
    o = out.float().cpu().numpy().reshape(-1, out.shape[-1]).astype(np.float64)
    l = lse.cpu().numpy().reshape(-1).astype(np.float64)
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        o, l = o[rows], l[rows]
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    err = np.abs(o - ref_out)
    tol = OUT_ATOL + OUT_RTOL * np.abs(ref_out) + P_E4M3_REL * bound
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} outputs out of tolerance, "
                           f"max err {err.max():.3e}")
    both_inf = np.isneginf(l) & np.isneginf(ref_lse)
    with np.errstate(invalid="ignore"):
        lerr = np.where(both_inf, 0.0, np.abs(l - ref_lse))
    assert np.all(lerr <= LSE_ATOL), f"{what}: lse max err {np.nanmax(lerr):.3e}"
    return float(err.max()), float(lerr.max())
