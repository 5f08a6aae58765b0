"""The decode's output bits depend only on its inputs.

The split plan and the persistent schedule are functions of the histories and
the grid shape (TokenSpeed AgentX post, "Balance MLA work with per-request KV
splitting": the split counts adapt to the current histories), partial states
are merged in a fixed order, and no state carries over from one call to the
next.  So the 1st and the 50th call of a process, the same call in two fresh
processes, and two different decodes running concurrently on two streams all
give the same bits (and match the oracle).
"""
import hashlib
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from helpers import SCALE, assert_parity, gpu_decode, oracle_decode, sample_rows, to_device
from paged_latent_attention_gb300 import api, inputs

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# A mixed batch: histories from one tile to several pages, so that the schedule
# has many segments and requests split across CTAs.
LENGTHS = [1, 127, 128, 1537, 9000, 33000, 200, 70_000, 12_345, 5, 2048, 40_000] * 4

CHILD = r"""
import hashlib, sys, torch
sys.path.insert(0, sys.argv[1])
from paged_latent_attention_gb300 import api, inputs
lens = [int(x) for x in sys.argv[2].split(",")]
w = inputs.custom_workload(lens, 1, 64, seed=77)
qn, qr, gate = inputs.make_queries(w, "cuda")
slab = inputs.make_slab(w, "cuda")
table = torch.as_tensor(w.page_table, device="cuda")
seq = torch.as_tensor(w.seq_lens, device="cuda")
out, lse = api.mla_decode(qn, qr, gate, slab, table, seq, n_q=1)
torch.cuda.synchronize()
h = hashlib.sha256()
h.update(out.view(torch.int16).cpu().numpy().tobytes())
h.update(lse.cpu().numpy().tobytes())
print(h.hexdigest())
"""


def _digest(out, lse):
    h = hashlib.sha256()
    h.update(out.view(torch.int16).cpu().numpy().tobytes())
    h.update(lse.cpu().numpy().tobytes())
    return h.hexdigest()


def _problem():
    w = inputs.custom_workload(LENGTHS, 1, 64, seed=77)
    qn, qr, gate = inputs.make_queries(w, "cuda")
    slab = inputs.make_slab(w, "cuda")
    table = torch.as_tensor(w.page_table, device="cuda")
    lens = torch.as_tensor(w.seq_lens, device="cuda")
    return w, qn, qr, gate, slab, table, lens


def test_first_and_fiftieth_call_give_the_same_bits():
    w, qn, qr, gate, slab, table, lens = _problem()
    ws = api.allocate_workspace(w.num_reqs, 1, 64)
    first_out, first_lse = api.mla_decode(qn, qr, gate, slab, table, lens, workspace=ws)
    first_out, first_lse = first_out.clone(), first_lse.clone()
    out = torch.empty_like(first_out)
    lse = torch.empty_like(first_lse)
    for _ in range(49):
        api.mla_decode(qn, qr, gate, slab, table, lens, workspace=ws, out=out, lse=lse)
    torch.cuda.synchronize()
    assert api.device_status(ws) == 0
    assert torch.equal(out.view(torch.int16), first_out.view(torch.int16))
    assert torch.equal(lse, first_lse)


def test_fresh_processes_give_the_same_bits():
    w, qn, qr, gate, slab, table, lens = _problem()
    out, lse = api.mla_decode(qn, qr, gate, slab, table, lens)
    mine = _digest(out, lse)
    arg = ",".join(str(int(x)) for x in LENGTHS)
    for _ in range(2):
        res = subprocess.run([sys.executable, "-c", CHILD, ROOT, arg], capture_output=True,
                             text=True, timeout=600, cwd=ROOT)
        assert res.returncode == 0, res.stderr[-2000:]
        assert res.stdout.strip().splitlines()[-1] == mine


def test_concurrent_decodes_of_different_shapes_on_two_streams():
    """A single-token decode and a 4-draft verify step run at the same time on
    two streams, each with its own workspace: both match the oracle and equal
    their results when run alone."""
    wa = inputs.custom_workload([20_000, 3000, 77, 15_000] * 4, 1, 64, seed=81)
    wb = inputs.custom_workload([9000, 4, 2500, 31_000, 600] * 3, 4, 64, seed=82)
    probs = []
    for w in (wa, wb):
        qn, qr, gate = inputs.make_queries(w, "cpu")
        slab = inputs.make_slab(w, "cpu", poison_nan=True)
        probs.append((w, (qn, qr, gate, slab), to_device(w, qn, qr, gate, slab)))
    alone = [gpu_decode(w, d) for (w, _, d) in probs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    wss = [api.allocate_workspace(w.num_reqs, w.n_q, w.num_heads) for (w, _, _) in probs]
    res = []
    torch.cuda.synchronize()
    for (w, _, d), s, ws in zip(probs, streams, wss):
        with torch.cuda.stream(s):
            res.append(api.mla_decode(d["qn"], d["qr"], d["gate"], d["slab"], d["table"],
                                      d["lens"], n_q=w.n_q, scale=SCALE, workspace=ws,
                                      stream=s))
    torch.cuda.synchronize()
    for ws in wss:
        assert api.device_status(ws) == 0
    for (w, host, _), (out, lse), (a_out, a_lse) in zip(probs, res, alone):
        assert torch.equal(out.view(torch.int16), a_out.view(torch.int16))
        assert torch.equal(lse, a_lse)
        rows = sample_rows(w, heads_per_token=6, seed=3)
        ref_out, ref_lse = oracle_decode(w, *host, rows=rows)
        assert_parity(out, lse, ref_out, ref_lse, rows=rows, what=f"concurrent n_q={w.n_q}")
