"""mla_decode_static_scratch: the decode entry point for callers that cannot
allocate device memory (an engine that reserved the device's memory for its page
pool, a plugin inside a framework that owns the allocator, a loop that cannot
take cudaMalloc's synchronisation).  It must give the same results as
mla_decode with a caller-provided workspace, call after call, although every
call reuses one scratch array compiled into the library.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from paged_latent_attention_gb300 import _native, api, inputs

pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(192.0)


def _inputs(lengths, n_q, H, seed):
    w = inputs.custom_workload(lengths, n_q, H, seed=seed, spare_pages=2)
    qn, qr, gate = inputs.make_queries(w, "cuda")
    slab = inputs.make_slab(w, "cuda", poison_nan=True)
    table = torch.as_tensor(w.page_table, device="cuda")
    lens = torch.as_tensor(w.seq_lens, device="cuda")
    return w, qn, qr, gate, slab, table, lens


def _static_scratch_call(w, qn, qr, gate, slab, table, lens, out, lse):
    stream = torch.cuda.current_stream().cuda_stream
    return _native.lib().mla_decode_static_scratch(
        qn.data_ptr(), qr.data_ptr(), gate.data_ptr(), slab.data_ptr(), slab.shape[0],
        slab.stride(0), table.data_ptr(), table.stride(0), lens.data_ptr(), w.num_reqs, w.n_q,
        w.num_heads, ctypes.c_float(SCALE), out.data_ptr(), lse.data_ptr(), 0, 1,
        stream if stream else None)


def _assert_close(out, lse, ref_out, ref_lse):
    o, r = out.float().cpu().numpy(), ref_out.float().cpu().numpy()
    assert np.all(np.abs(o - r) <= 1e-2 + 1e-2 * np.abs(r))
    l, rl = lse.cpu().numpy(), ref_lse.cpu().numpy()
    same_inf = np.isneginf(l) & np.isneginf(rl)
    with np.errstate(invalid="ignore"):
        assert np.all(same_inf | (np.abs(l - rl) <= 1e-3))


def test_static_scratch_matches_workspace_entry_point_on_consecutive_calls():
    cases = [([3000, 17000, 1, 9000], 1, 64, 31), ([5000, 130, 2], 4, 16, 32)]
    for lengths, n_q, H, seed in cases:          # two different calls in a row
        w, qn, qr, gate, slab, table, lens = _inputs(lengths, n_q, H, seed)
        ref_out, ref_lse = api.mla_decode(qn, qr, gate, slab, table, lens, n_q=n_q, scale=SCALE)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        status = _static_scratch_call(w, qn, qr, gate, slab, table, lens, out, lse)
        assert status == 0, _native.strerror(status)
        torch.cuda.synchronize()
        _assert_close(out, lse, ref_out, ref_lse)


def test_static_scratch_rejects_shapes_beyond_its_size():
    # 128 requests x 4 drafts x 64 heads needs far more than the 32 MiB array
    need = api.mla_workspace_size(128, 4, 64)
    assert need > (32 << 20)
    w, qn, qr, gate, slab, table, lens = _inputs([100] * 128, 4, 64, 33)
    out = torch.empty_like(qn)
    lse = torch.empty(qn.shape[0], 64, dtype=torch.float32, device="cuda")
    status = _static_scratch_call(w, qn, qr, gate, slab, table, lens, out, lse)
    assert status == 3 and _native.strerror(status) == "PLMLA_WORKSPACE_TOO_SMALL"
