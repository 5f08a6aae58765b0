"""A decode step captured once in a CUDA graph and replayed with new inputs.

The step plans its splits on the device from the lengths it reads at run time,
so one captured graph stays valid while histories change from step to step (no
host round trip per step; AgentX - InferenceXv3 report, SGLang section).  Each
replay here runs on new queries, gates and (shorter) histories written in place
into the captured buffers, and must match the oracle on those inputs.
"""
import copy

import numpy as np
import pytest
import torch

from helpers import SCALE, assert_parity, oracle_decode, sample_rows, to_device
from paged_latent_attention_gb300 import api, inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n_q,H", [(1, 64), (4, 16)])
def test_captured_step_follows_new_lengths_and_queries(n_q, H):
    lengths = [9000, 17000, 1, 4100, 30000, 1537]
    w = inputs.custom_workload(lengths, n_q, H, seed=70 + n_q, spare_pages=3)
    qn, qr, gate = inputs.make_queries(w, "cpu")
    slab = inputs.make_slab(w, "cpu", poison_nan=False)   # rows past a shortened history are read by nobody
    d = to_device(w, qn, qr, gate, slab)
    ws = api.allocate_workspace(w.num_reqs, n_q, H, 0, 1, "cuda")
    out = torch.empty_like(d["qn"])
    lse = torch.empty(d["qn"].shape[0], H, dtype=torch.float32, device="cuda")

    def step():
        api.mla_decode(d["qn"], d["qr"], d["gate"], d["slab"], d["table"], d["lens"], n_q=n_q,
                       scale=SCALE, out=out, lse=lse, workspace=ws)

    for _ in range(3):                 # eager calls first (tensor maps, function attributes)
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    rng = np.random.Generator(np.random.PCG64(5))
    for trial in range(3):
        new_lens = np.array([rng.integers(min(n_q, L), L + 1) for L in w.seq_lens], dtype=np.int32)
        g = torch.Generator().manual_seed(100 + trial)
        nq = torch.randn(qn.shape, generator=g).bfloat16()
        nr = torch.randn(qr.shape, generator=g).bfloat16()
        ng = torch.randn(gate.shape, generator=g).bfloat16()
        d["qn"].copy_(nq)
        d["qr"].copy_(nr)
        d["gate"].copy_(ng)
        d["lens"].copy_(torch.as_tensor(new_lens))
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert api.device_status(ws) == 0, "a decode pipeline wait timed out"
        w2 = copy.copy(w)
        w2.seq_lens = new_lens
        rows = sample_rows(w2, heads_per_token=4, seed=trial)
        ref_out, ref_lse = oracle_decode(w2, nq, nr, ng, slab, rows=rows)
        assert_parity(out, lse, ref_out, ref_lse, rows=rows, what=f"graph replay {trial}")


def test_captured_fp8_step_follows_new_queries():
    """The E4M3 step (its plan grid also quantises the queries) replays the same way."""
    from helpers import assert_parity_fp8, oracle_decode_fp8
    kvs = inputs.KV_SCALE_E4M3
    w = inputs.custom_workload([12000, 3000, 25000], 1, 64, seed=77, spare_pages=3)
    qn, qr, gate = inputs.make_queries(w, "cpu")
    slab = inputs.make_slab_e4m3(w, "cpu", poison_nan=False, kv_scale=kvs)
    d = to_device(w, qn, qr, gate, slab)
    ws = api.allocate_workspace(w.num_reqs, 1, 64, 0, 1, "cuda", fp8=True)
    out = torch.empty_like(d["qn"])
    lse = torch.empty(d["qn"].shape[0], 64, dtype=torch.float32, device="cuda")

    def step():
        api.mla_decode_fp8(d["qn"], d["qr"], d["gate"], d["slab"], d["table"], d["lens"],
                           kv_scale=kvs, n_q=1, scale=SCALE, out=out, lse=lse, workspace=ws)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    rng = np.random.Generator(np.random.PCG64(9))
    for trial in range(2):
        new_lens = np.array([rng.integers(1, L + 1) for L in w.seq_lens], dtype=np.int32)
        g = torch.Generator().manual_seed(200 + trial)
        nq = torch.randn(qn.shape, generator=g).bfloat16()
        nr = torch.randn(qr.shape, generator=g).bfloat16()
        ng = torch.randn(gate.shape, generator=g).bfloat16()
        d["qn"].copy_(nq)
        d["qr"].copy_(nr)
        d["gate"].copy_(ng)
        d["lens"].copy_(torch.as_tensor(new_lens))
        graph.replay()
        torch.cuda.synchronize()
        assert api.device_status(ws) == 0, "a decode pipeline wait timed out"
        w2 = copy.copy(w)
        w2.seq_lens = new_lens
        rows = sample_rows(w2, heads_per_token=4, seed=trial)
        ref_out, ref_lse, bound = oracle_decode_fp8(w2, nq, nr, ng, slab, kvs, rows=rows)
        assert_parity_fp8(out, lse, ref_out, ref_lse, bound, rows=rows, what=f"fp8 replay {trial}")
