"""Host logic of decode context parallelism (CPU, gloo, world sizes 2 and 3).

Each rank takes the pages of every request that the GPU path gives it (page
column c of request r belongs to rank (c + r) mod world), computes its gated
partial state with the oracle (the merge of its pages' one-page windows), and
the ranks all-gather and merge; the merge of the gated parts must equal the
oracle on the whole history (the gate is elementwise and the same for every
part, so gated parts merge directly)."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SCALE = 1.0 / np.sqrt(192.0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem():
    from paged_latent_attention_gb300 import inputs
    w = inputs.custom_workload([5000, 0, 1, 3100, 1536 * 2], 1, 16, seed=90, spare_pages=2)
    qn, qr, gate = inputs.make_queries(w, "cpu")
    slab = inputs.make_slab(w, "cpu")
    return w, qn, qr, gate, slab


def _attend(w, qn, qr, slab, t_lo=0, t_hi=None):
    import oracle
    return oracle.attend_rows(qn, qr, slab, w.page_table, w.seq_lens, 1, w.num_heads, SCALE,
                              num_pages=w.num_pages, t_lo=t_lo, t_hi=t_hi, threads=2)


def _rank_part(w, qn, qr, slab, rank, world):
    """The oracle's partial state of `rank`'s pages: its one-page windows merged."""
    import oracle
    from paged_latent_attention_gb300 import dcp
    rows_req = np.arange(w.num_reqs * w.num_heads) // w.num_heads
    os_, ls_ = [], []
    for c in range(w.page_table.shape[1]):
        o, lse = _attend(w, qn, qr, slab, c * 1536, (c + 1) * 1536)
        mine = np.array([dcp.owner(c, int(r), world) == rank for r in rows_req])
        os_.append(o)
        ls_.append(np.where(mine, lse, -np.inf))
    return oracle.lse_merge(np.stack(os_), np.stack(ls_))


def _worker(rank, world, port, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import oracle
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, qn, qr, gate, slab = _problem()
    o, lse = _rank_part(w, qn, qr, slab, rank, world)
    g = np.asarray(gate.float().numpy(), dtype=np.float64).reshape(o.shape)
    part = torch.from_numpy(oracle.gate_sigmoid(o, g))
    parts = [torch.empty_like(part) for _ in range(world)]
    lses = [torch.empty(lse.shape, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(parts, part)
    dist.all_gather(lses, torch.from_numpy(lse))
    out, lse_all = oracle.lse_merge(np.stack([p.numpy() for p in parts]),
                                    np.stack([l.numpy() for l in lses]))
    results[rank] = (out, lse_all)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3, 5])
def test_two_ranks_gather_and_merge_to_the_whole_history(world):
    """world 5: the short histories have fewer pages than ranks, so some ranks
    hold no token of a request and contribute empty parts (lse = -inf, weight 0)."""
    sys.path.insert(0, ROOT)
    import oracle
    port = _free_port()
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    w, qn, qr, gate, slab = _problem()
    o, lse = _attend(w, qn, qr, slab)
    g = np.asarray(gate.float().numpy(), dtype=np.float64).reshape(o.shape)
    ref = oracle.gate_sigmoid(o, g)
    for rank in range(world):
        out, lse_all = res[rank]
        np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
        both = np.isneginf(lse_all) & np.isneginf(lse)
        np.testing.assert_allclose(np.where(both, 0, lse_all), np.where(both, 0, lse),
                                   rtol=0, atol=1e-12)


@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_pages_cover_each_history_once_and_balance_the_ranks(world):
    """Host logic of the page-to-rank rule on the steady mix (64 histories in
    [8192, 32768]): every token belongs to exactly one rank, each request's
    ranks differ by at most one page, and the ranks' totals by a few pages."""
    sys.path.insert(0, ROOT)
    from paged_latent_attention_gb300 import dcp, inputs
    w = inputs.make_workload("steady")
    per = np.zeros((w.num_reqs, world), dtype=np.int64)
    for r, L in enumerate(w.seq_lens):
        for c in range(-(-int(L) // 1536)):
            per[r, dcp.owner(c, r, world)] += min(1536, int(L) - c * 1536)
    assert np.array_equal(per.sum(axis=1), w.seq_lens.astype(np.int64))
    assert (per.max(axis=1) - per.min(axis=1)).max() <= 1536
    totals = per.sum(axis=0)
    assert totals.max() - totals.min() <= 6 * 1536
    # the contiguous split it replaces left the ranks far apart
    if world > 1:
        assert totals.max() - totals.min() < 0.1 * totals.mean()
