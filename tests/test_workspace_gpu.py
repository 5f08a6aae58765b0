"""The workspace's contents on entry are irrelevant: a step must not read anything
it did not write in the same call.  Workspaces filled with NaN bit patterns, and
one workspace reused across calls of different shapes, give results that match
the oracle."""
import numpy as np
import pytest
import torch

from helpers import (SCALE, assert_parity, assert_parity_fp8, oracle_decode, oracle_decode_fp8,
                     sample_rows, to_device)
from paged_latent_attention_gb300 import api, inputs

pytestmark = pytest.mark.gpu


def _setup(lengths, n_q, H, seed, fp8=False):
    w = inputs.custom_workload(lengths, n_q, H, seed=seed, spare_pages=3)
    qn, qr, gate = inputs.make_queries(w, "cpu")
    if fp8:
        slab = inputs.make_slab_e4m3(w, "cpu", poison_nan=True, kv_scale=inputs.KV_SCALE_E4M3)
    else:
        slab = inputs.make_slab(w, "cpu", poison_nan=True)
    return w, qn, qr, gate, slab, to_device(w, qn, qr, gate, slab)


@pytest.mark.parametrize("fp8", [False, True])
def test_nan_filled_workspace(fp8):
    w, qn, qr, gate, slab, d = _setup([7000, 1, 20000, 1536, 3001], 1, 64, seed=95, fp8=fp8)
    ws = api.allocate_workspace(w.num_reqs, 1, 64, 0, 1, "cuda", fp8=fp8)
    ws.fill_(0xFF)                       # every fp32 / int32 word reads as NaN / -1
    kw = dict(n_q=1, scale=SCALE, workspace=ws)
    if fp8:
        out, lse = api.mla_decode_fp8(d["qn"], d["qr"], d["gate"], d["slab"], d["table"],
                                      d["lens"], kv_scale=inputs.KV_SCALE_E4M3, **kw)
    else:
        out, lse = api.mla_decode(d["qn"], d["qr"], d["gate"], d["slab"], d["table"], d["lens"],
                                  **kw)
    torch.cuda.synchronize()
    assert api.device_status(ws) == 0
    rows = sample_rows(w, heads_per_token=4, seed=5)
    if fp8:
        ref_out, ref_lse, bound = oracle_decode_fp8(w, qn, qr, gate, slab, inputs.KV_SCALE_E4M3,
                                                    rows=rows)
        assert_parity_fp8(out, lse, ref_out, ref_lse, bound, rows=rows, what="NaN workspace fp8")
    else:
        ref_out, ref_lse = oracle_decode(w, qn, qr, gate, slab, rows=rows)
        assert_parity(out, lse, ref_out, ref_lse, rows=rows, what="NaN workspace")


def test_one_workspace_across_shapes():
    """A workspace sized for the largest call, reused by calls of other shapes in
    turn (more requests, draft tokens, fewer heads), each leaving its state behind."""
    shapes = [([9000, 4000, 15000, 2], 1, 64, 96), ([3000, 12000], 4, 16, 97),
              ([2, 5000, 2500, 8000, 700, 30000], 2, 32, 98), ([9000, 4000, 15000, 2], 1, 64, 96)]
    size = max(api.mla_workspace_size(len(L), n_q, H, 0, 1) for L, n_q, H, _ in shapes)
    ws = torch.full((size,), 0xFF, dtype=torch.uint8, device="cuda")
    for i, (lengths, n_q, H, seed) in enumerate(shapes):
        w, qn, qr, gate, slab, d = _setup(lengths, n_q, H, seed)
        out, lse = api.mla_decode(d["qn"], d["qr"], d["gate"], d["slab"], d["table"], d["lens"],
                                  n_q=n_q, scale=SCALE, workspace=ws)
        torch.cuda.synchronize()
        assert api.device_status(ws) == 0
        rows = sample_rows(w, heads_per_token=4, seed=i)
        ref_out, ref_lse = oracle_decode(w, qn, qr, gate, slab, rows=rows)
        assert_parity(out, lse, ref_out, ref_lse, rows=rows, what=f"shape {i}")
        assert np.isfinite(out.float().cpu().numpy()).all()
