"""Decode context parallelism on one GPU: the ranks' parts run one after the
other here (each is an ordinary mla_decode on the rank's pages, from
mla_dcp_shard; no kernel waits on another), then mla_merge_partials merges them
as the exchange step would.  The merged result must match the oracle on the
whole history, and mla_decode on the whole history."""
import numpy as np
import pytest
import torch

from helpers import SCALE, assert_parity, gpu_decode, oracle_decode, to_device
from paged_latent_attention_gb300 import api, dcp, inputs

pytestmark = pytest.mark.gpu


def _parts(w, d, world):
    outs, lses = [], []
    for rank in range(world):
        table_k, lens_k = dcp.shard_view(d["table"], d["lens"], rank, world)
        out, lse = api.mla_decode(d["qn"], d["qr"], d["gate"], d["slab"], table_k, lens_k,
                                  n_q=1, scale=SCALE)
        outs.append(out)
        lses.append(lse)
    return torch.stack(outs).contiguous(), torch.stack(lses).contiguous()


@pytest.mark.parametrize("world", [1, 2, 3, 5])
def test_ranks_parts_merge_to_the_whole_history(world):
    # histories of 0, 1, a few pages, and ones that end inside a rank's first page
    lengths = [7000, 0, 1, 1536 * 3, 20000, 1537, 12345]
    w = inputs.custom_workload(lengths, 1, 64, seed=80 + world, spare_pages=3)
    qn, qr, gate = inputs.make_queries(w, "cpu")
    slab = inputs.make_slab(w, "cpu", poison_nan=True)
    d = to_device(w, qn, qr, gate, slab)
    out_parts, lse_parts = _parts(w, d, world)
    out, lse = api.mla_merge_partials(out_parts, lse_parts)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle_decode(w, qn, qr, gate, slab)
    assert_parity(out, lse, ref_out, ref_lse, what=f"dcp world={world}")
    whole_out, whole_lse = gpu_decode(w, d)
    torch.testing.assert_close(out.float(), whole_out.float(), atol=2e-2, rtol=2e-2)
    finite = torch.isfinite(whole_lse)
    assert torch.equal(finite, torch.isfinite(lse))
    torch.testing.assert_close(lse[finite], whole_lse[finite], atol=1e-3, rtol=0)


@pytest.mark.parametrize("world", [2, 3])
def test_fp8_pages_parts_merge_to_the_whole_history(world):
    """E4M3 pages: each rank's part carries the E4M3 probability rounding of its
    own tokens; weighted by exp(lse_k - lse), those errors add up to the same
    bound as one decode over the whole history."""
    from helpers import assert_parity_fp8, oracle_decode_fp8
    kvs = inputs.KV_SCALE_E4M3
    lengths = [9000, 1, 1536 * 2, 16000, 0]
    w = inputs.custom_workload(lengths, 1, 64, seed=90 + world, spare_pages=3)
    qn, qr, gate = inputs.make_queries(w, "cpu")
    slab = inputs.make_slab_e4m3(w, "cpu", poison_nan=True, kv_scale=kvs)
    d = to_device(w, qn, qr, gate, slab)
    outs, lses = [], []
    for rank in range(world):
        o, l = dcp.decode_shard(d["qn"], d["qr"], d["gate"], d["slab"], d["table"], d["lens"],
                                rank, world, kv_scale=kvs, scale=SCALE)
        outs.append(o)
        lses.append(l)
    out, lse = api.mla_merge_partials(torch.stack(outs).contiguous(),
                                      torch.stack(lses).contiguous())
    torch.cuda.synchronize()
    ref_out, ref_lse, bound = oracle_decode_fp8(w, qn, qr, gate, slab, kvs)
    assert_parity_fp8(out, lse, ref_out, ref_lse, bound, what=f"fp8 dcp world={world}")


def test_merge_of_one_part_is_that_part_and_no_part_is_empty():
    T, H = 3, 16
    g = torch.Generator(device="cuda").manual_seed(4)
    part = torch.randn(1, T, H, 512, device="cuda", generator=g).bfloat16()
    lse1 = torch.randn(1, T, H, device="cuda", generator=g)
    out, lse = api.mla_merge_partials(part, lse1)
    assert torch.equal(out, part[0]) and torch.equal(lse, lse1[0])
    empty = torch.full((2, T, H), float("-inf"), device="cuda")
    out, lse = api.mla_merge_partials(torch.stack([part[0], part[0]]).contiguous(), empty)
    assert torch.equal(out, torch.zeros_like(out)) and bool(torch.isneginf(lse).all())


def test_dcp_decode_through_a_one_rank_process_group():
    """dcp_decode end to end (view, decode, all-gather, merge) in a one-rank NCCL
    group: the collective path runs, and equals mla_decode on the whole history."""
    import socket

    import torch.distributed as dist
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    store = dist.TCPStore("127.0.0.1", port, 1, True)
    dist.init_process_group("nccl", store=store, rank=0, world_size=1)
    try:
        w = inputs.custom_workload([9000, 2, 4000], 1, 16, seed=85, spare_pages=2)
        qn, qr, gate = inputs.make_queries(w, "cpu")
        slab = inputs.make_slab(w, "cpu", poison_nan=True)
        d = to_device(w, qn, qr, gate, slab)
        out, lse = dcp.dcp_decode(d["qn"], d["qr"], d["gate"], d["slab"], d["table"], d["lens"],
                                  scale=SCALE)
        torch.cuda.synchronize()
        ref_out, ref_lse = oracle_decode(w, qn, qr, gate, slab)
        assert_parity(out, lse, ref_out, ref_lse, what="dcp_decode one rank")
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_shard_kernel_follows_the_page_rule(world):
    """mla_dcp_shard against the rule restated on the host: rank k's row holds
    the page IDs of the columns c with (c + r) mod world == k, in column order,
    and its length their tokens (the last page partial)."""
    from paged_latent_attention_gb300 import dcp
    rng = np.random.Generator(np.random.PCG64(70 + world))
    R, ld = 37, 23
    lens = rng.integers(0, ld * 1536 + 1, size=R).astype(np.int32)
    lens[:4] = [0, 1, 1536, 1537]
    table = rng.integers(0, 10_000, size=(R, ld + 5)).astype(np.int32)
    dt = torch.as_tensor(table, device="cuda")[:, :ld]          # row stride ld + 5
    dl = torch.as_tensor(lens, device="cuda")
    total = np.zeros(R, dtype=np.int64)
    for rank in range(world):
        tk, lk = api.mla_dcp_shard(dt, dl, world, rank)
        tk, lk = tk.cpu().numpy(), lk.cpu().numpy()
        for r in range(R):
            n = -(-int(lens[r]) // 1536)
            cols = [c for c in range(n) if dcp.owner(c, r, world) == rank]
            assert tk[r, :len(cols)].tolist() == [int(table[r, c]) for c in cols]
            expect = sum(min(1536, int(lens[r]) - c * 1536) for c in cols)
            assert int(lk[r]) == expect
            total[r] += expect
    assert np.array_equal(total, lens.astype(np.int64))
