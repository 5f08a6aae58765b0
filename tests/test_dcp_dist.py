"""Host logic of decode context parallelism (CPU, gloo, world sizes 2 and 3).

Each rank takes its token range of every request from the same page-table
column split the GPU path uses, computes its gated partial state with the
oracle, and the ranks all-gather and merge; the merge of the gated parts must
equal the oracle on the whole history (the gate is elementwise and the same for
every part, so gated parts merge directly)."""
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


def _worker(rank, world, port, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import oracle
    from paged_latent_attention_gb300 import dcp
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, qn, qr, gate, slab = _problem()
    t_lo, t_hi = dcp.shard_bounds(rank, world, w.page_table.shape[1])
    o, lse = _attend(w, qn, qr, slab, t_lo, t_hi)
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


@pytest.mark.parametrize("world", [2, 3])
def test_two_ranks_gather_and_merge_to_the_whole_history(world):
    """world 3: four table columns split 2 + 2 + 0, so the last rank holds no
    token of any request and contributes empty parts (lse = -inf, weight 0)."""
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


@pytest.mark.parametrize("world", [1, 2, 3, 4, 7])
def test_shard_view_lengths_cover_each_history_once(world):
    sys.path.insert(0, ROOT)
    from paged_latent_attention_gb300 import dcp
    lens = torch.tensor([0, 1, 1535, 1536, 1537, 9000, 20000], dtype=torch.int32)
    cols = 14
    table = torch.arange(7 * cols, dtype=torch.int32).reshape(7, cols)
    total = torch.zeros_like(lens)
    for rank in range(world):
        table_k, lens_k = dcp.shard_view(table, lens, rank, world)
        t_lo, t_hi = dcp.shard_bounds(rank, world, cols)
        assert table_k.stride() == table.stride()
        assert bool((lens_k >= 0).all()) and bool((lens_k <= t_hi - t_lo).all())
        live = lens_k > 0
        # a rank's first column is the page holding its first token
        if bool(live.any()):
            assert int(table_k[0, 0]) == int(table[0, t_lo // 1536])
        total += lens_k
    assert torch.equal(total, lens)
