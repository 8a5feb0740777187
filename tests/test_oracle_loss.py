"""Pins for the loss-boundary oracle (CPU): library routines on single
chains, closed forms, a hand-worked advantage example, GRPO as the one-group
special case, and invariants."""
import numpy as np
import pytest
import torch

from oracle import layout as OL
from oracle import loss as OLS
from workloads import trees as WT


def test_position_ids_closed_forms():
    t = WT.chain_tree([3, 4, 2])
    assert OLS.position_ids(t.parent, t.seg_len).tolist() == list(range(9))
    P, R = 5, [3, 1, 4]
    pos = OLS.position_ids([-1, 0, 0, 0], [P] + R)
    want = list(range(P)) + sum([list(range(P, P + r)) for r in R], [])
    assert pos.tolist() == want


def test_multiplicity_sums_to_expanded_tokens():
    rng = np.random.default_rng(5)
    for _ in range(10):
        t = WT.random_tree(rng, int(rng.integers(1, 9)), [1, 2, 5], n_roots=int(rng.integers(1, 3)))
        mult = OL.multiplicity(t.parent, t.seg_len)
        assert mult.sum() == t.n_expanded


def test_logprobs_chain_equals_torch_log_softmax():
    rng = np.random.default_rng(0)
    t = WT.chain_tree([6, 5])
    N, V = t.n_tokens, 37
    logits = rng.normal(size=(N, V)) * 3
    tokens = rng.integers(0, V, size=N)
    got = OLS.traj_logprobs(t.parent, t.seg_len, logits, tokens)
    ls = torch.log_softmax(torch.tensor(logits, dtype=torch.float64), dim=-1)
    want = ls[:-1].gather(1, torch.tensor(tokens[1:]).long()[:, None])[:, 0].numpy()
    assert np.abs(got - want).max() < 1e-12


def test_logprobs_star_branch_rows():
    # the last prompt row predicts each response's first token; shared rows agree
    rng = np.random.default_rng(1)
    P, R = 4, [3, 2]
    parent, seg = [-1, 0, 0], [P] + R
    N, V = sum(seg), 11
    logits = rng.normal(size=(N, V))
    tokens = rng.integers(0, V, size=N)
    lp = OLS.traj_logprobs(parent, seg, logits, tokens)
    n1 = P + R[0] - 1
    a, b = lp[:n1], lp[n1:]
    assert np.allclose(a[:P - 1], b[:P - 1], atol=0, rtol=0)
    lse = OLS.row_logsumexp(logits)
    assert abs(a[P - 1] - (logits[P - 1, tokens[P]] - lse[P - 1])) < 1e-12
    assert abs(b[P - 1] - (logits[P - 1, tokens[P + R[0]]] - lse[P - 1])) < 1e-12
    assert np.allclose(np.exp(logits - lse[:, None]).sum(axis=1), 1.0, atol=1e-12)


def test_advantage_hand_worked_binary_tree():
    # root 0 -> a 1, b 2; a -> leaves 3, 4; b -> leaves 5, 6; rewards [1, 0, 0, 0]
    parent, seg = [-1, 0, 0, 1, 1, 2, 2], [2, 1, 1, 1, 1, 1, 1]
    A, node_c, tok_c = OLS.subtree_advantage(parent, seg, [1, 0, 0, 0])
    # l3: (1 - .25 + 1 - .5) / 2; l4: (-.25 - .5) / 2; l5, l6: (-.25 + 0) / 2
    assert np.allclose(A, [0.625, -0.375, -0.125, -0.125], atol=1e-15)
    assert np.allclose(node_c, [0.0, 0.25, -0.25, 0.625, -0.375, -0.125, -0.125], atol=1e-15)
    A, _, _ = OLS.subtree_advantage(parent, seg, [1, 0, 0, 0], size_weighted=True)
    # l3: (4 * .75 + 2 * .5) / 6
    assert np.allclose(A[0], 4.0 / 6.0)
    A, _, _ = OLS.subtree_advantage(parent, seg, [1, 0, 0, 0], no_root=True)
    assert np.allclose(A, [0.5, -0.5, 0.0, 0.0])
    # token coefficients follow the packed order: root(2), a(1), l3, l4, b(1), l5, l6
    assert np.allclose(tok_c, [0, 0, 0.25, 0.625, -0.375, -0.25, -0.125, -0.125])


def test_advantage_single_group_is_grpo():
    rng = np.random.default_rng(2)
    r = rng.normal(size=8)
    parent = [-1] + [0] * 8
    A, _, _ = OLS.subtree_advantage(parent, [3] + [2] * 8, r, norm_std=True, eps=1e-6)
    assert np.allclose(A, (r - np.mean(r)) / (np.std(r) + 1e-6), atol=1e-13)


def test_advantage_invariants():
    rng = np.random.default_rng(3)
    t = WT.random_tree(rng, 12, [1, 2, 3], n_roots=2)
    L = len(OL.leaves(t.parent))
    r = rng.normal(size=L)
    A, nc, _ = OLS.subtree_advantage(t.parent, t.seg_len, r)
    A2, _, _ = OLS.subtree_advantage(t.parent, t.seg_len, r + 7.5)
    assert np.allclose(A, A2, atol=1e-12)                 # shift invariance
    A3, _, _ = OLS.subtree_advantage(t.parent, t.seg_len, 3 * r)
    assert np.allclose(A3, 3 * A, atol=1e-12)             # linear without normalisation
    roots = [u for u in range(len(t.parent)) if t.parent[u] < 0]
    assert np.isclose(sum(nc[u] for u in roots), A.sum())
