"""The uniform split rule on the GPU (the baseline of the TokenSpeed AgentX post's
Figure 5 comparison, section "Balance MLA work with per-request KV splitting"):
the device planner against the oracle's uniform baseline, bit for bit, including
the left panel of Figure 4; and the decode under that rule against the oracle.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_parity, gpu_decode, oracle_decode, to_device
from paged_latent_attention_gb300 import api, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture
def uniform_mode():
    api.set_split_mode("uniform")
    try:
        yield
    finally:
        api.set_split_mode("per-request")


def test_uniform_plan_matches_oracle(uniform_mode):
    golden = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                         "planner_fig4.json")))["cases"]
    cases = [(c["seq_lens"], c["budget"]) for c in golden]
    rng = np.random.Generator(np.random.PCG64(21))
    for _ in range(60):
        R = int(rng.integers(1, 1025))
        lens = rng.integers(0, 1_000_001, size=R)
        lens[rng.random(R) < 0.1] = 0
        cases.append((lens.tolist(), int(rng.integers(1, 4097))))
    cases.append(([0] * 5, 7))
    for lens, budget in cases:
        _, splits = oracle.plan_splits_uniform(lens, budget, 128)
        indptr, dchunk = api.mla_plan_splits(torch.tensor(lens, dtype=torch.int32,
                                                          device="cuda"), budget)
        expect = np.concatenate([[0], np.cumsum(splits)]).astype(np.int64)
        assert int(dchunk.item()) == 0
        assert np.array_equal(indptr.cpu().numpy().astype(np.int64), expect), (len(lens), budget)
    # Figure 4, left panel: 64k and 192k with 16 chunks -> 8 and 8
    indptr, _ = api.mla_plan_splits(torch.tensor([65536, 196608], dtype=torch.int32,
                                                 device="cuda"), 16)
    assert indptr.cpu().tolist() == [0, 8, 16]


@pytest.mark.parametrize("n_q,H,cta_budget", [(1, 64, 0), (4, 64, 0), (1, 16, 12), (3, 32, 0)])
def test_uniform_decode_matches_oracle(uniform_mode, n_q, H, cta_budget):
    lengths = [1, 127, 129, 1536, 1537, 40_000, 3000, 0, 90_000, 17]
    lengths = [max(L, n_q) if L else 0 for L in lengths]
    w = inputs.custom_workload(lengths, n_q, H, seed=600 + 7 * n_q + H, spare_pages=3)
    qn, qr, gate = inputs.make_queries(w, "cpu")
    slab = inputs.make_slab(w, "cpu", poison_nan=True)
    d = to_device(w, qn, qr, gate, slab)
    out, lse = gpu_decode(w, d, cta_budget=cta_budget)
    ref_out, ref_lse = oracle_decode(w, qn, qr, gate, slab)
    assert_parity(out, lse, ref_out, ref_lse, what=f"uniform n_q={n_q} H={H}")
