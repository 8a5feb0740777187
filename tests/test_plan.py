"""The library's C++ planner, called through the C ABI, against the
brute-force plan of the oracle (dense ancestor mask): bit-exact (CPU only)."""
import json
import os

import numpy as np
import pytest

from oracle import layout as OL
from oracle import plan as OP
from prefix_tree_attention_attn_gb300 import TreePlan
from workloads import trees as WT

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiny_binary_plan.json")


def lib_plan(t, block, chunk=0):
    p = TreePlan(t.parent, t.seg_len, block=block, bwd_chunk_qtiles=chunk)
    return p, p.export()


def compare(t, block, qtiles=None, chunk=0):
    p, e = lib_plan(t, block, chunk)
    ref = OP.brute_plan(t.parent, t.seg_len, block=block, qtiles=qtiles)
    N, T = ref["N"], ref["T"]
    assert p.n_tokens == N and p.info["n_qtiles"] == T
    assert list(e["node_order"]) == list(ref["node_order"])
    assert list(e["node_off"]) == list(ref["node_off"])
    tiles = range(T) if qtiles is None else qtiles
    for t_ in tiles:
        a, b = e["qi_ptr"][t_], e["qi_ptr"][t_ + 1]
        got_iv = list(zip(e["qi_lo"][a:b].tolist(), e["qi_hi"][a:b].tolist()))
        assert got_iv == ref["intervals"][t_], t_
        a, b = e["qt_ptr"][t_], e["qt_ptr"][t_ + 1]
        got = list(zip(e["qt_kv"][a:b].tolist(), e["qt_cls"][a:b].tolist()))
        assert got == ref["tiles"][t_], t_
    if qtiles is None:
        np.testing.assert_array_equal(e["subend"], ref["subend"])
        assert list(zip(e["kv_qlo"].tolist(), e["kv_qhi"].tolist())) == ref["kv_range"]
        assert p.n_pairs == OP.pair_count(t.parent, t.seg_len)
        assert p.info["n_tile_entries"] == sum(len(v) for v in ref["tiles"].values())
        assert p.info["n_full_tiles"] == sum(1 for v in ref["tiles"].values() for _, c in v if c == OP.FULL)
    check_schedules(p, e)
    return p, e


def check_schedules(p, e):
    T = p.info["n_qtiles"]
    cost = np.diff(e["qt_ptr"])
    order = e["fwd_order"]
    assert sorted(order.tolist()) == list(range(T))
    assert all(cost[order[k]] >= cost[order[k + 1]] for k in range(T - 1))
    items = e["bwd_items"].reshape(-1, 4)
    S = p.info["bwd_chunk_qtiles"]
    covered = {}
    slots = set()
    for c, t0, t1, slot in items.tolist():
        assert e["kv_qlo"][c] <= t0 < t1 <= e["kv_qhi"][c]
        covered.setdefault(c, []).append((t0, t1))
        if slot >= 0:
            assert slot not in slots
            slots.add(slot)
    assert len(slots) == p.info["n_partial_slots"]
    for c in range(T):
        segs = sorted(covered[c])
        assert segs[0][0] == e["kv_qlo"][c] and segs[-1][1] == e["kv_qhi"][c]
        assert all(segs[k][1] == segs[k + 1][0] for k in range(len(segs) - 1))
    # q-ranges are cut at multiples of S; items run chunk by chunk, longest first within
    assert all((t0 // S) == ((t1 - 1) // S) for _, t0, t1, _ in items.tolist())
    keys = [(t0 // S, -(t1 - t0)) for _, t0, t1, _ in items.tolist()]
    assert keys == sorted(keys)


def test_golden_tiny_tree():
    g = json.load(open(GOLDEN))
    t = WT.Tree("g", g["parent"], g["seg_len"])
    for block in (128, 64):
        p, e = compare(t, block)
        exp = g[f"block{block}"]
        T = p.info["n_qtiles"]
        ivs = [[[int(a), int(b)] for a, b in zip(e["qi_lo"][e["qi_ptr"][k]:e["qi_ptr"][k + 1]],
                                                 e["qi_hi"][e["qi_ptr"][k]:e["qi_ptr"][k + 1]])]
               for k in range(T)]
        assert ivs == exp["intervals"]
    assert p.n_pairs == g["pairs"]


def all_small_trees(max_nodes):
    import itertools
    for n in range(1, max_nodes + 1):
        for par in itertools.product(range(-1, n), repeat=n):
            if any(par[v] == v for v in range(n)):
                continue
            ok = True
            for v in range(n):
                u, s = v, 0
                while par[u] >= 0 and s <= n:
                    u = par[u]
                    s += 1
                if s > n:
                    ok = False
                    break
            if ok:
                yield list(par)


def test_all_small_forests_small_tiles():
    rng = np.random.default_rng(3)
    count = 0
    for par in all_small_trees(4):
        lens = [int(x) for x in rng.choice([1, 2, 3, 7], size=len(par))]
        t = WT.Tree("s", par, lens)
        for block in (1, 2, 3, 4):
            compare(t, block)
        count += 1
    assert count > 100


@pytest.mark.parametrize("seed", range(30))
def test_random_forests(seed):
    rng = np.random.default_rng(1000 + seed)
    n = int(rng.integers(1, 40))
    t = WT.random_tree(rng, n, [1, 2, 3, 5, 8, 13, 127, 128, 129], n_roots=1 + seed % 4)
    block = [1, 4, 7, 16, 32, 128][seed % 6]
    compare(t, block, chunk=int(rng.integers(0, 4)))


@pytest.mark.parametrize("name", ["tiny_binary", "grpo_star", "segment_tree", "agentic_tree"])
def test_workload_trees_full(name):
    t = WT.load_tree(name)
    compare(t, 128)


def test_long_context_sampled_tiles():
    t = WT.load_tree("long_context")
    p = TreePlan(t.parent, t.seg_len)
    T = p.info["n_qtiles"]
    rng = np.random.default_rng(5)
    qtiles = sorted(set(rng.choice(T, size=24, replace=False).tolist()) | {0, T - 1})
    compare(t, 128, qtiles=qtiles)
    e = p.export(["subend", "node_off"])
    # subend from the definition on sampled keys: last attending query + 1
    tn = OL.token_nodes(t.parent, t.seg_len)
    A = OL.ancestor_matrix(t.parent)
    N = p.n_tokens
    for j in rng.choice(N, size=40, replace=False):
        u = tn[j]
        rows = np.nonzero(A[tn, u] & ((tn != u) | (np.arange(N) >= j)))[0]
        assert rows[0] == j and rows[-1] + 1 == e["subend"][j] and rows.size == e["subend"][j] - j


def test_chain_merge_gives_identical_token_plan():
    a = TreePlan([-1, 0, 1], [100, 200, 57]).export()
    b = TreePlan([-1], [357]).export()
    for f in ("subend", "qi_ptr", "qi_lo", "qi_hi", "qt_ptr", "qt_kv", "qt_cls", "kv_qlo", "kv_qhi"):
        np.testing.assert_array_equal(a[f], b[f])


def expected_chunk(e, T):
    """The automatic backward chunk as include/tree_attn.h states it: 24 q-tiles
    below 64 q-tiles, 48 below 256, else 64, doubled while the kv-tiles whose
    q-range spans several chunks would need more than max(2048, 8 T) slots."""
    lo, hi = e["kv_qlo"].astype(np.int64), e["kv_qhi"].astype(np.int64)

    def slots(S):
        n = (hi - 1) // S - lo // S + 1
        return int(n[n > 1].sum())

    S = 24 if T < 64 else (48 if T < 256 else 64)
    while S < T and slots(S) > max(2048, 8 * T):
        S *= 2
    return S


@pytest.mark.parametrize("name", ["tiny_binary", "segment_tree", "grpo_star", "agentic_tree", "long_context",
                                  "chain"])
def test_automatic_chunk_rule(lib, name):
    t = WT.chain_tree([2048 * 128]) if name == "chain" else WT.load_tree(name)
    p = TreePlan(t.parent, t.seg_len)
    e = p.export(("kv_qlo", "kv_qhi"))
    T = p.info["n_qtiles"]
    assert p.info["bwd_chunk_qtiles"] == expected_chunk(e, T)
    if name == "chain":        # 2,048 q-tiles of one chain: the slot cap doubles the chunk
        assert p.info["bwd_chunk_qtiles"] > 64
