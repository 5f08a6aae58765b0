"""mla_decode_static_scratch: the decode entry point for callers that cannot
allocate device memory (an engine that reserved the device's memory for its page
pool, a plugin inside a framework that owns the allocator, a loop that cannot
take cudaMalloc's synchronisation).  Every call reuses one scratch array
compiled into the library, so these tests check consecutive calls of different
shapes -- one just under the array's size, then a smaller one that finds the
larger call's leftovers in the array -- against the oracle, and bit for bit
against mla_decode with a workspace of its own (the schedule depends only on
the inputs, so both give the same bits).  The step's status word is read
through mla_static_scratch_status after every call.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from helpers import SCALE, assert_parity, oracle_decode, sample_rows
from paged_latent_attention_gb300 import _native, api, inputs

pytestmark = pytest.mark.gpu

LIMIT = 32 << 20          # PLMLA_STATIC_SCRATCH_BYTES


def _inputs(lengths, n_q, H, seed):
    w = inputs.custom_workload(lengths, n_q, H, seed=seed, spare_pages=2)
    qn, qr, gate = inputs.make_queries(w, "cpu")
    slab = inputs.make_slab(w, "cpu", poison_nan=True)
    dev = dict(qn=qn.cuda(), qr=qr.cuda(), gate=gate.cuda(), slab=slab.cuda(),
               table=torch.as_tensor(w.page_table, device="cuda"),
               lens=torch.as_tensor(w.seq_lens, device="cuda"))
    return w, (qn, qr, gate, slab), dev


def _stream():
    s = torch.cuda.current_stream().cuda_stream
    return s if s else None


def _static_scratch_call(w, d, out, lse):
    return _native.lib().mla_decode_static_scratch(
        d["qn"].data_ptr(), d["qr"].data_ptr(), d["gate"].data_ptr(), d["slab"].data_ptr(),
        d["slab"].shape[0], d["slab"].stride(0), d["table"].data_ptr(), d["table"].stride(0),
        d["lens"].data_ptr(), w.num_reqs, w.n_q, w.num_heads, ctypes.c_float(SCALE),
        out.data_ptr(), lse.data_ptr(), 0, 1, _stream())


def _status():
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rc = _native.lib().mla_static_scratch_status(ctypes.c_void_p(st.data_ptr()), _stream())
    assert rc == 0, _native.strerror(rc)
    torch.cuda.synchronize()
    return int(st.item())


def _requests_near_limit(n_q, H):
    """The largest request count whose workspace fits the array, and its size."""
    best = None
    for R in range(1, 1025):
        need = api.mla_workspace_size(R, n_q, H)
        if need > LIMIT:
            break
        best = (R, need)
    return best


def _check_call(w, host, d, what):
    out = torch.full((w.num_tokens, w.num_heads, 512), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    lse = torch.full((w.num_tokens, w.num_heads), float("nan"), device="cuda")
    rc = _static_scratch_call(w, d, out, lse)
    assert rc == 0, _native.strerror(rc)
    torch.cuda.synchronize()
    assert _status() == 0, f"{what}: the step's status word is set"
    # the oracle on sampled rows (every request, heads 0, H-1 and two more)
    rows = sample_rows(w, heads_per_token=4, seed=7)
    ref_out, ref_lse = oracle_decode(w, *host, rows=rows)
    assert_parity(out, lse, ref_out, ref_lse, rows=rows, what=what)
    # and bit for bit the workspace entry point
    ws_out, ws_lse = api.mla_decode(d["qn"], d["qr"], d["gate"], d["slab"], d["table"],
                                    d["lens"], n_q=w.n_q, scale=SCALE)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ws_out.view(torch.int16)), what
    assert torch.equal(lse, ws_lse), what


def test_static_scratch_matches_oracle_on_consecutive_calls():
    R, need = _requests_near_limit(1, 64)
    assert need > LIMIT - (1 << 20), "the near-limit case should fill the array"
    rng = np.random.Generator(np.random.PCG64(41))
    big = [int(x) for x in rng.integers(1, 2400, size=R)]
    big[0] = 1537                       # one request crosses a page boundary
    cases = [(big, 1, 64, 41), ([5000, 130, 2], 4, 16, 42), ([3000, 17000, 1, 9000], 1, 64, 43)]
    for lengths, n_q, H, seed in cases:       # three calls in a row, large shape first
        assert api.mla_workspace_size(len(lengths), n_q, H) <= LIMIT
        w, host, d = _inputs(lengths, n_q, H, seed)
        _check_call(w, host, d, f"static scratch R={len(lengths)} n_q={n_q} H={H}")


def test_static_scratch_rejects_shapes_beyond_its_size():
    R, _ = _requests_near_limit(1, 64)
    assert api.mla_workspace_size(R + 1, 1, 64) > LIMIT
    for lengths, n_q in (([100] * (R + 1), 1), ([100] * 128, 4)):
        w, _, d = _inputs(lengths, n_q, 64, 44)
        out = torch.empty(w.num_tokens, 64, 512, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(w.num_tokens, 64, dtype=torch.float32, device="cuda")
        rc = _static_scratch_call(w, d, out, lse)
        assert rc == 3 and _native.strerror(rc) == "PLMLA_WORKSPACE_TOO_SMALL"
