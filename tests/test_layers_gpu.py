"""mla_decode_layers: the decode step of several MLA layers that share one page
table (TokenSpeed Kimi K3 post, section "A Generic, Unified Flat KV Layout for
Cache Management": each slab holds one MLA page per global page ID, so the
layers differ only in their slab).  The split plan is made once for the step;
every layer must give mla_decode's bits for its own tensors, and match the
oracle.  Also: E4M3 slabs with one scale per layer, lse for some layers only,
and the layered step captured in a CUDA graph and replayed with new lengths.
"""
import copy

import numpy as np
import pytest
import torch

from helpers import (SCALE, assert_parity, assert_parity_fp8, oracle_decode, oracle_decode_fp8,
                     sample_rows)
from paged_latent_attention_gb300 import api, inputs

pytestmark = pytest.mark.gpu

LENGTHS = [1, 127, 128, 1537, 9000, 20_000, 3, 4099, 640, 33_000]


def _layers(w, L, poison=True):
    host = []
    for l in range(L):
        qn, qr, gate = inputs.make_queries(w, "cpu", layer=l)
        slab = inputs.make_slab(w, "cpu", layer=l, poison_nan=poison)
        host.append((qn, qr, gate, slab))
    dev = [tuple(t.cuda() for t in h) for h in host]
    return host, dev


@pytest.mark.parametrize("n_q,H", [(1, 64), (4, 64), (2, 16)])
def test_layers_equal_single_layer_calls_and_the_oracle(n_q, H):
    L = 3
    w = inputs.custom_workload(LENGTHS, n_q, H, seed=500 + n_q + H, spare_pages=2)
    host, dev = _layers(w, L)
    table = torch.as_tensor(w.page_table, device="cuda")
    lens = torch.as_tensor(w.seq_lens, device="cuda")
    ws = api.allocate_workspace(w.num_reqs, n_q, H, 0, 1, "cuda")
    outs, lses = api.mla_decode_layers([d[0] for d in dev], [d[1] for d in dev],
                                       [d[2] for d in dev], [d[3] for d in dev], table, lens,
                                       n_q=n_q, scale=SCALE, workspace=ws)
    torch.cuda.synchronize()
    assert api.device_status(ws) == 0
    rows = sample_rows(w, heads_per_token=4, seed=9)
    for l in range(L):
        one_out, one_lse = api.mla_decode(*dev[l][:3], dev[l][3], table, lens, n_q=n_q,
                                          scale=SCALE)
        torch.cuda.synchronize()
        assert torch.equal(outs[l].view(torch.int16), one_out.view(torch.int16)), l
        assert torch.equal(lses[l], one_lse), l
        ref_out, ref_lse = oracle_decode(w, *host[l], rows=rows)
        assert_parity(outs[l], lses[l], ref_out, ref_lse, rows=rows, what=f"layer {l}")


def test_layers_fp8_with_a_scale_per_layer():
    L, n_q, H = 3, 1, 64
    w = inputs.custom_workload(LENGTHS, n_q, H, seed=611, spare_pages=2)
    scales = [6.0 / 448.0, 3.0 / 448.0, 12.0 / 448.0]
    host, dev = [], []
    for l in range(L):
        qn, qr, gate = inputs.make_queries(w, "cpu", layer=l)
        slab8 = inputs.make_slab_e4m3(w, "cpu", layer=l, poison_nan=True, kv_scale=scales[l])
        host.append((qn, qr, gate, slab8))
        dev.append((qn.cuda(), qr.cuda(), gate.cuda(), slab8.cuda()))
    table = torch.as_tensor(w.page_table, device="cuda")
    lens = torch.as_tensor(w.seq_lens, device="cuda")
    outs, lses = api.mla_decode_layers([d[0] for d in dev], [d[1] for d in dev],
                                       [d[2] for d in dev], [d[3] for d in dev], table, lens,
                                       n_q=n_q, scale=SCALE, kv_scale=scales)
    torch.cuda.synchronize()
    rows = sample_rows(w, heads_per_token=4, seed=10)
    for l in range(L):
        one_out, one_lse = api.mla_decode_fp8(*dev[l][:3], dev[l][3], table, lens,
                                              kv_scale=scales[l], n_q=n_q, scale=SCALE)
        torch.cuda.synchronize()
        assert torch.equal(outs[l].view(torch.int16), one_out.view(torch.int16)), l
        assert torch.equal(lses[l], one_lse), l
        ref_out, ref_lse, terms = oracle_decode_fp8(w, *host[l], scales[l], rows=rows)
        assert_parity_fp8(outs[l], lses[l], ref_out, ref_lse, terms, rows=rows,
                          what=f"fp8 layer {l}")


def test_layers_lse_for_some_layers_only():
    L, n_q, H = 2, 1, 16
    w = inputs.custom_workload([700, 5000, 1], n_q, H, seed=620, spare_pages=1)
    host, dev = _layers(w, L)
    table = torch.as_tensor(w.page_table, device="cuda")
    lens = torch.as_tensor(w.seq_lens, device="cuda")
    lse1 = torch.full((w.num_tokens, H), float("nan"), device="cuda")
    outs, lses = api.mla_decode_layers([d[0] for d in dev], [d[1] for d in dev],
                                       [d[2] for d in dev], [d[3] for d in dev], table, lens,
                                       n_q=n_q, scale=SCALE, lse=[None, lse1])
    torch.cuda.synchronize()
    assert lses[0] is None and lses[1] is lse1
    # layer 0 without LSE: the same output bits as a single-layer call
    one_out, _ = api.mla_decode(*dev[0][:3], dev[0][3], table, lens, n_q=n_q, scale=SCALE)
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), one_out.view(torch.int16))
    ref_out, ref_lse = oracle_decode(w, *host[1])
    assert_parity(outs[1], lse1, ref_out, ref_lse, what="layer 1")


def test_captured_layered_step_follows_new_lengths():
    L, n_q, H = 4, 1, 64
    lengths = [9000, 17000, 1, 4100, 30000, 1537]
    w = inputs.custom_workload(lengths, n_q, H, seed=630, spare_pages=3)
    host, dev = _layers(w, L, poison=False)   # rows past a shortened history are read by nobody
    table = torch.as_tensor(w.page_table, device="cuda")
    lens = torch.as_tensor(w.seq_lens, device="cuda")
    ws = api.allocate_workspace(w.num_reqs, n_q, H, 0, 1, "cuda")
    outs = [torch.empty_like(d[0]) for d in dev]
    lses = [torch.empty(w.num_tokens, H, device="cuda") for _ in range(L)]

    def step():
        api.mla_decode_layers([d[0] for d in dev], [d[1] for d in dev], [d[2] for d in dev],
                              [d[3] for d in dev], table, lens, n_q=n_q, scale=SCALE, out=outs,
                              lse=lses, workspace=ws)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    rng = np.random.Generator(np.random.PCG64(6))
    for trial in range(2):
        new_lens = np.array([rng.integers(1, L_ + 1) for L_ in w.seq_lens], dtype=np.int32)
        lens.copy_(torch.as_tensor(new_lens))
        for o in outs:
            o.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert api.device_status(ws) == 0
        w2 = copy.copy(w)
        w2.seq_lens = new_lens
        rows = sample_rows(w2, heads_per_token=3, seed=trial)
        for l in (0, L - 1):
            ref_out, ref_lse = oracle_decode(w2, *host[l], rows=rows)
            assert_parity(outs[l], lses[l], ref_out, ref_lse, rows=rows,
                          what=f"replay {trial} layer {l}")


def test_one_layer_equals_mla_decode():
    w = inputs.custom_workload([3000, 17, 9000], 2, 64, seed=640, spare_pages=1)
    host, dev = _layers(w, 1)
    table = torch.as_tensor(w.page_table, device="cuda")
    lens = torch.as_tensor(w.seq_lens, device="cuda")
    outs, lses = api.mla_decode_layers([dev[0][0]], [dev[0][1]], [dev[0][2]], [dev[0][3]], table,
                                       lens, n_q=2, scale=SCALE)
    one_out, one_lse = api.mla_decode(*dev[0][:3], dev[0][3], table, lens, n_q=2, scale=SCALE)
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), one_out.view(torch.int16))
    assert torch.equal(lses[0], one_lse)


def test_layers_under_the_uniform_split_rule():
    """The uniform baseline of the pages' Figure 5 plans the step once for every
    layer too: each layer equals its single-layer call under the same rule."""
    L = 2
    w = inputs.custom_workload([20_000, 300, 7000, 1537], 1, 64, seed=650, spare_pages=2)
    host, dev = _layers(w, L)
    table = torch.as_tensor(w.page_table, device="cuda")
    lens = torch.as_tensor(w.seq_lens, device="cuda")
    api.set_split_mode("uniform")
    try:
        outs, lses = api.mla_decode_layers([d[0] for d in dev], [d[1] for d in dev],
                                           [d[2] for d in dev], [d[3] for d in dev], table, lens,
                                           n_q=1, scale=SCALE)
        singles = [api.mla_decode(*d[:3], d[3], table, lens, n_q=1, scale=SCALE) for d in dev]
        torch.cuda.synchronize()
    finally:
        api.set_split_mode("per-request")
    rows = sample_rows(w, heads_per_token=4, seed=11)
    for l in range(L):
        assert torch.equal(outs[l].view(torch.int16), singles[l][0].view(torch.int16)), l
        assert torch.equal(lses[l], singles[l][1]), l
        ref_out, ref_lse = oracle_decode(w, *host[l], rows=rows)
        assert_parity(outs[l], lses[l], ref_out, ref_lse, rows=rows, what=f"uniform layer {l}")


def test_page_check_covers_the_layered_step():
    """With page checks on, one check after the layered step reports a table
    entry outside the pool (status 40); requests that do not use it keep their
    results in every layer."""
    L = 2
    lengths = [4000, 9000, 3000]
    w = inputs.custom_workload(lengths, 1, 64, seed=660, spare_pages=2)
    host, dev = _layers(w, L, poison=False)
    table_np = w.page_table.copy()
    table_np[1, (lengths[1] - 1) // inputs.PAGE_TOKENS] = w.num_pages + 5
    table = torch.as_tensor(table_np, device="cuda")
    lens = torch.as_tensor(w.seq_lens, device="cuda")
    ws = api.allocate_workspace(w.num_reqs, 1, 64, 0, 1, "cuda")
    api.set_page_checks(True)
    try:
        outs, lses = api.mla_decode_layers([d[0] for d in dev], [d[1] for d in dev],
                                           [d[2] for d in dev], [d[3] for d in dev], table, lens,
                                           n_q=1, scale=SCALE, workspace=ws)
        torch.cuda.synchronize()
    finally:
        api.set_page_checks(False)
    assert api.device_status(ws) == 40
    rows = sample_rows(w, heads_per_token=4, seed=12)
    good = rows[rows // w.num_heads != 1]
    for l in range(L):
        ref_out, ref_lse = oracle_decode(w, *host[l], rows=good)
        assert_parity(outs[l], lses[l], ref_out, ref_lse, rows=good, what=f"good requests, layer {l}")
