"""Pins for the batching oracle (CPU): closed forms, hand-worked LPT
examples, Graham's bound against the brute-force optimum, and invariants."""
import itertools

import numpy as np
import pytest

from oracle import batch as OB
from oracle import layout as OL
from workloads import trees as WT


def test_pairs_chain_closed_form():
    # a chain of segments is one causal sequence of L tokens: L (L + 1) / 2 pairs
    for lens in ([1], [5], [3, 4], [2, 2, 2, 7]):
        t = WT.chain_tree(lens)
        L = sum(lens)
        assert OB.pairs_by_walking(t.parent, t.seg_len) == L * (L + 1) // 2


def test_pairs_star_closed_form():
    # prompt P with responses R_i: P(P+1)/2 + sum_i R_i (R_i + 1) / 2 + R_i P
    P, R = 7, [3, 1, 6]
    parent = [-1] + [0] * len(R)
    want = P * (P + 1) // 2 + sum(r * (r + 1) // 2 + r * P for r in R)
    assert OB.pairs_by_walking(parent, [P] + R) == want


def test_pairs_equal_sum_of_positions():
    # each token attends its own position + 1 tokens along its path; the
    # positions are taken here from the expanded trajectories
    rng = np.random.default_rng(3)
    for _ in range(20):
        t = WT.random_tree(rng, int(rng.integers(1, 9)), [1, 2, 3, 5], n_roots=int(rng.integers(1, 3)))
        _, off, N = OL.packed_layout(t.parent, t.seg_len)
        pos = [None] * N
        for _, idx in OL.trajectories(t.parent, t.seg_len):
            for p, tok in enumerate(idx):
                assert pos[tok] in (None, p)
                pos[tok] = p
        assert OB.pairs_by_walking(t.parent, t.seg_len) == sum(p + 1 for p in pos)


def test_pairs_forest_additive():
    a, b = WT.chain_tree([3, 2]), WT.Tree("s", [-1, 0, 0], [4, 1, 2])
    par, seg, src = OB.forest([(a.parent, a.seg_len), (b.parent, b.seg_len)], [True, True])
    assert src == [0, 0, 1, 1, 1]
    assert OB.pairs_by_walking(par, seg) == OB.pairs_by_walking(a.parent, a.seg_len) + \
        OB.pairs_by_walking(b.parent, b.seg_len)


def test_lpt_hand_worked():
    # 10->r0, 8->r1, 7->r1 (8 < 10), 6->r0 (10 < 15), 5->r1 (15 < 16), 4->r0 (16 < 20)
    rep, load = OB.lpt([10, 8, 7, 6, 5, 4], 2)
    assert rep == [0, 1, 1, 0, 1, 0] and load == [20, 20]
    # ties: equal work in index order, equal loads to the lowest replica
    rep, load = OB.lpt([5, 5, 5], 2)
    assert rep == [0, 1, 0] and load == [10, 5]
    rep, load = OB.lpt([1, 9, 4], 5)
    assert rep == [2, 0, 1] and load == [9, 4, 1, 0, 0]


@pytest.mark.parametrize("seed", range(30))
def test_lpt_within_graham_bound(seed):
    rng = np.random.default_rng(seed)
    n, R = int(rng.integers(1, 8)), int(rng.integers(1, 4))
    work = [int(x) for x in rng.integers(0, 50, size=n)]
    _, load = OB.lpt(work, R)
    best = min(max(sum(w for w, r in zip(work, a) if r == q) for q in range(R))
               for a in itertools.product(range(R), repeat=n))
    assert sum(load) == sum(work)
    assert max(load) * 3 * R <= (4 * R - 1) * best or max(load) == best


def test_microbatches_hand_worked():
    work = [9, 1, 5, 7, 3]
    toks = [6, 2, 5, 4, 3]
    rep = [0, 0, 1, 0, 0]
    # replica 0 in LPT order: tree 0 (6 tok) -> mb0, tree 3 (4) -> mb1 (6+4 > 8), tree 4 (3) -> mb1? 4+3 = 7 <= 8,
    # tree 1 (2) -> mb0 (6+2 = 8)
    mb, n = OB.microbatches(work, toks, rep, 0, 8)
    assert mb == [0, 0, -1, 1, 1] and n == 2
    mb, n = OB.microbatches(work, toks, rep, 1, 3)   # tree 2 is above the cap: alone
    assert mb == [-1, -1, 0, -1, -1] and n == 1
