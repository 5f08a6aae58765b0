"""The opt-in page-table check that runs after a decode step.

A page ID is only ever a coordinate of the slab's tensor map, so an ID outside
the pool reads zeros instead of faulting and the step's output is silently
wrong; with checks on, the step's status word says so (40), and a history that
needs more columns than the table row holds is reported too (41).  Requests
whose pages are good keep their exact results.
"""
import numpy as np
import pytest
import torch

from helpers import SCALE, assert_parity, oracle_decode, sample_rows, to_device
from paged_latent_attention_gb300 import api, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture
def checks_on():
    api.set_page_checks(True)
    try:
        yield
    finally:
        api.set_page_checks(False)


def _setup(lengths, seed):
    w = inputs.custom_workload(lengths, 1, 64, seed=seed, spare_pages=2)
    qn, qr, gate = inputs.make_queries(w, "cpu")
    slab = inputs.make_slab(w, "cpu", poison_nan=False)
    return w, qn, qr, gate, slab


def _decode(w, d):
    ws = api.allocate_workspace(w.num_reqs, 1, 64, 0, 1, "cuda")
    out, lse = api.mla_decode(d["qn"], d["qr"], d["gate"], d["slab"], d["table"], d["lens"],
                              n_q=1, scale=SCALE, workspace=ws)
    torch.cuda.synchronize()
    return out, lse, api.device_status(ws)


def test_switch_defaults_off_and_toggles():
    assert api.get_page_checks() is False
    api.set_page_checks(True)
    try:
        assert api.get_page_checks() is True
    finally:
        api.set_page_checks(False)
    assert api.get_page_checks() is False


def test_good_table_passes_with_checks_on(checks_on):
    w, qn, qr, gate, slab = _setup([5000, 1, 1536, 1537, 20000], seed=81)
    d = to_device(w, qn, qr, gate, slab)
    out, lse, status = _decode(w, d)
    assert status == 0
    rows = sample_rows(w, heads_per_token=4, seed=1)
    ref_out, ref_lse = oracle_decode(w, qn, qr, gate, slab, rows=rows)
    assert_parity(out, lse, ref_out, ref_lse, rows=rows, what="checked step")


@pytest.mark.parametrize("bad", ["past_pool", "negative"])
def test_out_of_range_page_is_reported(checks_on, bad):
    lengths = [4000, 9000, 3000]
    w, qn, qr, gate, slab = _setup(lengths, seed=82)
    table = w.page_table.copy()
    # the last used column of request 1: a coordinate the tensor map reads as zeros
    table[1, (lengths[1] - 1) // inputs.PAGE_TOKENS] = w.num_pages + 3 if bad == "past_pool" else -1
    d = to_device(w, qn, qr, gate, slab)
    d["table"].copy_(torch.as_tensor(table))
    out, lse, status = _decode(w, d)
    assert status == 40
    # requests 0 and 2 use none of the bad entry: their results stand
    rows = sample_rows(w, heads_per_token=4, seed=2)
    good = rows[rows // w.num_heads != 1]          # one token per request: row = r * H + h
    assert good.size
    ref_out, ref_lse = oracle_decode(w, qn, qr, gate, slab, rows=good)
    assert_parity(out, lse, ref_out, ref_lse, rows=good, what="requests with good pages")


def test_bad_entry_past_the_history_is_not_reported(checks_on):
    """Columns past ceil(L / 1536) are never read, whatever they hold."""
    lengths = [1536, 2000]
    w, qn, qr, gate, slab = _setup(lengths, seed=83)
    assert w.page_table.shape[1] >= 2
    table = w.page_table.copy()
    table[0, 1:] = -7                      # request 0 uses column 0 only
    d = to_device(w, qn, qr, gate, slab)
    d["table"].copy_(torch.as_tensor(table))
    out, lse, status = _decode(w, d)
    assert status == 0
    rows = sample_rows(w, heads_per_token=4, seed=3)
    ref_out, ref_lse = oracle_decode(w, qn, qr, gate, slab, rows=rows)
    assert_parity(out, lse, ref_out, ref_lse, rows=rows, what="unused bad columns")


def test_history_longer_than_the_row_is_reported(checks_on):
    """Request 0 claims one page more than its row holds: the step reads that
    column from the start of row 1 (inside the table buffer) and the check says 41."""
    lengths = [3000, 3000, 3000]
    w, qn, qr, gate, slab = _setup(lengths, seed=84)
    ld = w.page_table.shape[1]
    lens = np.array(w.seq_lens, dtype=np.int32)
    lens[0] = ld * inputs.PAGE_TOKENS + 5
    d = to_device(w, qn, qr, gate, slab)
    d["lens"].copy_(torch.as_tensor(lens))
    _, _, status = _decode(w, d)
    assert status == 41


def test_checks_off_leaves_status_clear():
    lengths = [4000, 9000]
    w, qn, qr, gate, slab = _setup(lengths, seed=85)
    table = w.page_table.copy()
    table[1, 0] = w.num_pages + 1
    d = to_device(w, qn, qr, gate, slab)
    d["table"].copy_(torch.as_tensor(table))
    _, _, status = _decode(w, d)
    assert status == 0
