"""Pins for the oracle's split planner (CPU only).

The pages print one worked example (TokenSpeed AgentX post, section "Balance MLA
work with per-request KV splitting", Figure 4 and its equal-length control); it is
stored with its citation in tests/golden/planner_fig4.json.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "planner_fig4.json")


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases())
def test_figure4_worked_example(case):
    chunk, splits = oracle.plan_splits(case["seq_lens"], case["budget"], case["tile"])
    assert chunk == case["expect_chunk"]
    assert splits == case["expect_splits"]
    assert sum(splits) == case["budget"]
    # every chunk has the same length in the worked example
    for L, s in zip(case["seq_lens"], splits):
        assert L == s * chunk
    if "uniform_splits" in case:
        per_req = case["budget"] // len(case["seq_lens"])
        assert [per_req] * len(case["seq_lens"]) == case["uniform_splits"]
        assert [L // per_req for L in case["seq_lens"]] == case["uniform_chunk_lens"]
        # per-request splitting shortens the longest chunk (the kernel's tail)
        assert chunk < max(case["uniform_chunk_lens"])
        # the oracle's uniform baseline gives the figure's left panel exactly
        # (tile 1: the figure's chunks are not rounded)
        uchunks, usplits = oracle.plan_splits_uniform(case["seq_lens"], case["budget"], 1)
        assert usplits == case["uniform_splits"]
        assert uchunks == case["uniform_chunk_lens"]


def test_equal_length_control_keeps_total_work():
    cases = _cases()
    mixed, control = cases[0], cases[2]
    assert sum(control["seq_lens"]) == sum(mixed["seq_lens"])
    assert len(set(control["seq_lens"])) == 1


def test_longer_requests_get_more_splits():
    rng = np.random.Generator(np.random.PCG64(0))
    for _ in range(200):
        R = int(rng.integers(1, 40))
        lens = rng.integers(0, 300_000, size=R).tolist()
        budget = int(rng.integers(1, 600))
        chunk, splits = oracle.plan_splits(lens, budget, 128)
        order = np.argsort(lens, kind="stable")
        assert all(splits[order[i]] <= splits[order[i + 1]] for i in range(R - 1))
        assert chunk % 128 == 0
        for L, s in zip(lens, splits):
            assert s == (0 if L == 0 else -(-L // chunk))
            if L > 0:
                assert (s - 1) * chunk < L <= s * chunk


def test_budget_is_respected_when_possible_and_chunk_is_smallest():
    rng = np.random.Generator(np.random.PCG64(1))
    for _ in range(300):
        R = int(rng.integers(1, 20))
        lens = rng.integers(1, 100_000, size=R).tolist()
        budget = int(rng.integers(1, 200))
        tile = int(rng.choice([64, 128]))
        chunk, splits = oracle.plan_splits(lens, budget, tile)
        longest = -(-max(lens) // tile) * tile
        assert sum(splits) <= budget or all(s == 1 for s in splits)
        assert chunk <= max(longest, -(-(-(-sum(lens) // budget)) // tile) * tile)
        start = -(-(-(-sum(lens) // budget)) // tile) * tile
        assert chunk >= start
        if chunk > start:   # the next smaller candidate did not fit
            smaller = chunk - tile
            assert sum(-(-L // smaller) for L in lens) > budget


def test_more_requests_than_budget_gives_one_split_each():
    chunk, splits = oracle.plan_splits([5000] * 10 + [70_000], 4, 128)
    assert splits == [1] * 11 and chunk == 70_016


def test_empty_requests_get_no_split():
    assert oracle.plan_splits([0, 0], 8, 128) == (128, [0, 0])
    chunk, splits = oracle.plan_splits([0, 1000, 0], 8, 128)
    assert splits[0] == 0 and splits[2] == 0 and splits[1] >= 1


def test_uniform_baseline_rounds_to_the_tile_and_keeps_the_split_count():
    rng = np.random.Generator(np.random.PCG64(2))
    for _ in range(200):
        R = int(rng.integers(1, 40))
        lens = rng.integers(0, 300_000, size=R).tolist()
        budget = int(rng.integers(1, 600))
        chunks, splits = oracle.plan_splits_uniform(lens, budget, 128)
        live = sum(1 for L in lens if L > 0)
        su = max(1, budget // max(1, live))
        for L, c, s in zip(lens, chunks, splits):
            if L == 0:
                assert (c, s) == (0, 0)
                continue
            assert c % 128 == 0 and (s - 1) * c < L <= s * c
            assert s <= su                           # rounding up never adds a split
            assert c - 128 < -(-L // su) <= c        # the smallest tile multiple that fits
        assert sum(splits) <= max(budget, live)
