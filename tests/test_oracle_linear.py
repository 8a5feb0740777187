"""Pins for the tree linear-attention oracle (CPU): the parallel and the
recurrent formula agree; a single chain with no decay equals causal
(QK^T masked) V computed with torch; copies agree across trajectories; a
pure-Python brute force on tiny trees."""
import numpy as np
import pytest
import torch

from oracle import layout as OL
from oracle import linear as OLN
from workloads import trees as WT


def rnd(N, hq, hkv, d, seed):
    g = np.random.default_rng(seed)
    return g.normal(size=(N, hq, d)), g.normal(size=(N, hkv, d)), g.normal(size=(N, hkv, d))


def test_chain_no_decay_equals_masked_matmul():
    t = WT.chain_tree([5, 7])
    q, k, v = rnd(t.n_tokens, 2, 1, 4, 0)
    o = OLN.forward_parallel(t.parent, t.seg_len, q, k, v, [1.0], 0.5)
    Q, K, V = (torch.tensor(x, dtype=torch.float64) for x in (q, k, v))
    s = Q[:, 0] @ K[:, 0].T
    want = 0.5 * (torch.tril(s) @ V[:, 0])
    assert np.abs(o[:, 0] - want.numpy()).max() < 1e-12


@pytest.mark.parametrize("seed", range(4))
def test_parallel_equals_recurrent_on_trees(seed):
    rng = np.random.default_rng(seed)
    t = WT.random_tree(rng, int(rng.integers(2, 8)), [1, 2, 4], n_roots=int(rng.integers(1, 3)))
    q, k, v = rnd(t.n_tokens, 4, 2, 3, seed)
    dec = [0.9, 1.0]
    a = OLN.forward_parallel(t.parent, t.seg_len, q, k, v, dec, 0.7)
    b = OLN.forward_recurrent(t.parent, t.seg_len, q, k, v, dec, 0.7)
    assert np.isfinite(a).all() and np.abs(a - b).max() < 1e-11


def test_brute_force_tiny_tree():
    parent, seg = [-1, 0, 0], [2, 1, 2]
    t = WT.Tree("t", parent, seg)
    q, k, v = rnd(t.n_tokens, 1, 1, 2, 7)
    gam = 0.8
    o = OLN.forward_parallel(parent, seg, q, k, v, [gam], 1.0)
    _, off, N = OL.packed_layout(parent, seg)
    # by hand: each token's path in packed order, positions 0.. along it
    paths = {0: [0], 1: [0, 1], 2: [0, 1, 2], 3: [0, 1, 3], 4: [0, 1, 3, 4]}
    for i, path in paths.items():
        pi = len(path) - 1
        want = sum(gam ** (pi - pj) * float(q[i, 0] @ k[j, 0]) * v[j, 0] for pj, j in enumerate(path))
        assert np.abs(o[i, 0] - want).max() < 1e-12


def test_copies_agree_and_shared_prefix_equals_chain():
    # the prompt of a star gets the same output as the prompt alone
    t = WT.Tree("s", [-1, 0, 0], [6, 3, 4])
    q, k, v = rnd(t.n_tokens, 2, 1, 3, 3)
    o = OLN.forward_parallel(t.parent, t.seg_len, q, k, v, [0.95], 1.0)
    c = WT.chain_tree([6])
    oc = OLN.forward_parallel(c.parent, c.seg_len, q[:6], k[:6], v[:6], [0.95], 1.0)
    assert np.abs(o[:6] - oc).max() < 1e-12
