"""Teams of query rows that share KV loads (thread-block clusters with TMA
multicast; include/plmla.h, mla_set_team_clusters).

When a step's query rows form two or more teams of 64 (several draft tokens, or
128 heads) of at most 8 members each, the CTAs holding the same member's work
for 2 or 4 teams run as one cluster and each KV tile is loaded once for all of
them.  Only the loads change, so every cluster width must give the same bits,
and match the oracle -- on ragged histories whose pages past each history hold
NaN, with the default grid (many members per team: no clusters) and a small one
of 16 CTAs (2 to 8 members per team: clusters of 2, or 4 when the width allows
it and the team count divides).
"""
import pytest
import torch

from helpers import SCALE, assert_parity, gpu_decode, oracle_decode, sample_rows, to_device
from paged_latent_attention_gb300 import api, inputs

pytestmark = pytest.mark.gpu

LENGTHS = [1, 127, 128, 129, 1535, 1536, 1537, 4099, 20_000, 3, 9000, 640]


@pytest.fixture
def restore_width():
    try:
        yield
    finally:
        api.set_team_clusters(2)


@pytest.mark.parametrize("n_q,H", [(4, 64), (2, 64), (1, 128), (8, 64)])
@pytest.mark.parametrize("cta_budget", [0, 16])
def test_every_cluster_width_gives_the_same_bits(restore_width, n_q, H, cta_budget):
    w = inputs.custom_workload(LENGTHS, n_q, H, seed=300 + 11 * n_q + H, spare_pages=2)
    qn, qr, gate = inputs.make_queries(w, "cpu")
    slab = inputs.make_slab(w, "cpu", poison_nan=True)
    d = to_device(w, qn, qr, gate, slab)
    results = {}
    for width in (1, 2, 4):
        api.set_team_clusters(width)
        results[width] = gpu_decode(w, d, cta_budget=cta_budget)
    out1, lse1 = results[1]
    for width in (2, 4):
        out, lse = results[width]
        assert torch.equal(out.view(torch.int16), out1.view(torch.int16)), width
        assert torch.equal(lse, lse1), width
    rows = sample_rows(w, heads_per_token=6, seed=5)
    ref_out, ref_lse = oracle_decode(w, qn, qr, gate, slab, rows=rows)
    assert_parity(out1, lse1, ref_out, ref_lse, rows=rows, what=f"clusters n_q={n_q} H={H}")
