"""Pins for the brute-force plan (CPU): the hand-derived tiny-tree fixture, and
the subtree-contiguity lemma the library's planner relies on."""
import json
import os

import numpy as np
import pytest

from oracle import layout as OL
from oracle import plan as OP
from workloads import trees as WT

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiny_binary_plan.json")


def load_golden():
    with open(GOLDEN) as f:
        return json.load(f)


def test_golden_layout_and_subend():
    g = load_golden()
    p = OP.brute_plan(g["parent"], g["seg_len"], block=128)
    assert p["N"] == g["n_tokens"]
    assert list(p["node_order"]) == g["node_order"]
    assert list(p["node_off"]) == g["node_off"]
    sub = np.zeros(g["n_tokens"], dtype=np.int64)
    for a, b, e in g["subend_runs"]:
        sub[a:b] = e
    np.testing.assert_array_equal(p["subend"], sub)
    assert OP.pair_count(g["parent"], g["seg_len"]) == g["pairs"]
    assert int(OL.dense_mask(g["parent"], g["seg_len"]).sum()) == g["pairs"]


@pytest.mark.parametrize("block", [128, 64])
def test_golden_tiles(block):
    g = load_golden()
    exp = g[f"block{block}"]
    p = OP.brute_plan(g["parent"], g["seg_len"], block=block)
    T = p["T"]
    assert [[list(x) for x in p["intervals"][t]] for t in range(T)] == exp["intervals"]
    assert [[list(x) for x in p["tiles"][t]] for t in range(T)] == exp["tiles"]
    assert [list(x) for x in p["kv_range"]] == exp["kv_range"]


@pytest.mark.parametrize("seed", range(40))
def test_lemma_queries_of_a_key_are_contiguous(seed):
    rng = np.random.default_rng(500 + seed)
    t = WT.random_tree(rng, int(rng.integers(1, 12)), [1, 2, 3, 5, 8], n_roots=1 + seed % 3)
    assert OP.key_query_sets_contiguous(t.parent, t.seg_len)
    M = OL.dense_mask(t.parent, t.seg_len)
    assert int(M.sum()) == OP.pair_count(t.parent, t.seg_len)
    # every q-tile between a kv-tile's first and last user is itself a user
    for B in (1, 2, 3, 4):
        p = OP.brute_plan(t.parent, t.seg_len, block=B)
        users = {c: [tt for tt in range(p["T"]) if any(cc == c for cc, _ in p["tiles"][tt])]
                 for c in range(p["T"])}
        for c, us in users.items():
            assert us == list(range(p["kv_range"][c][0], p["kv_range"][c][1]))
            assert us[0] == c
