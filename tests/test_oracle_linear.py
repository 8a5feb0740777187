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


# --------------------------------------------------------------------------
# backward: pinned by finite differences of the forward oracle (O is linear in
# each of Q, K and V, so central differences are exact up to rounding), the
# closed form of one token, and the invariance of the dO split over copies
# --------------------------------------------------------------------------

def _loss(t, q, k, v, do, dec, scale):
    return float((OLN.forward_parallel(t.parent, t.seg_len, q, k, v, dec, scale) * do).sum())


@pytest.mark.parametrize("tree", [([-1, 0, 0], [2, 2, 1]), ([-1, 0, 1, 0, -1], [1, 2, 1, 2, 2])])
def test_backward_equals_finite_differences(tree):
    t = WT.Tree("fd", *tree)
    N = t.n_tokens
    q, k, v = rnd(N, 4, 2, 2, 11)
    do = np.random.default_rng(12).normal(size=(N, 4, 2))
    dec, scale, eps = [0.8, 1.0], 0.6, 1e-3
    dq, dk, dv = OLN.backward_parallel(t.parent, t.seg_len, q, k, v, do, dec, scale)
    for x, g in ((q, dq), (k, dk), (v, dv)):
        fd = np.zeros_like(x)
        for ix in np.ndindex(*x.shape):
            keep = x[ix]
            x[ix] = keep + eps
            up = _loss(t, q, k, v, do, dec, scale)
            x[ix] = keep - eps
            dn = _loss(t, q, k, v, do, dec, scale)
            x[ix] = keep
            fd[ix] = (up - dn) / (2 * eps)
        assert np.abs(g - fd).max() <= 1e-8 * max(1.0, np.abs(fd).max())


def test_backward_one_token_closed_form():
    t = WT.chain_tree([1])
    q, k, v = rnd(1, 1, 1, 3, 5)
    do = np.random.default_rng(6).normal(size=(1, 1, 3))
    s = 0.9
    dq, dk, dv = OLN.backward_parallel(t.parent, t.seg_len, q, k, v, do, [0.5], s)
    qk, dov = float(q[0, 0] @ k[0, 0]), float(do[0, 0] @ v[0, 0])
    assert np.abs(dq[0, 0] - s * dov * k[0, 0]).max() < 1e-14
    assert np.abs(dk[0, 0] - s * dov * q[0, 0]).max() < 1e-14
    assert np.abs(dv[0, 0] - s * qk * do[0, 0]).max() < 1e-14


@pytest.mark.parametrize("seed", range(3))
def test_backward_split_invariance(seed):
    rng = np.random.default_rng(40 + seed)
    t = WT.random_tree(rng, int(rng.integers(3, 8)), [1, 2, 5], n_roots=1 + seed % 2)
    q, k, v = rnd(t.n_tokens, 2, 1, 3, seed)
    do = rng.normal(size=(t.n_tokens, 2, 3))
    a = OLN.backward_parallel(t.parent, t.seg_len, q, k, v, do, [0.9], 1.0, split="multiplicity")
    b = OLN.backward_parallel(t.parent, t.seg_len, q, k, v, do, [0.9], 1.0, split="first")
    for x, y in zip(a, b):
        assert np.abs(x - y).max() < 1e-11


@pytest.mark.parametrize("seed", range(4))
def test_backward_recurrent_equals_parallel(seed):
    """The adjoint recursion over compact tokens (no expansion) against the
    per-trajectory VJP with the dO split over copies."""
    rng = np.random.default_rng(60 + seed)
    t = WT.random_tree(rng, int(rng.integers(2, 9)), [1, 2, 3, 6], n_roots=1 + seed % 2)
    q, k, v = rnd(t.n_tokens, 4, 2, 3, seed)
    do = rng.normal(size=(t.n_tokens, 4, 3))
    dec = [0.85, 1.0]
    a = OLN.backward_parallel(t.parent, t.seg_len, q, k, v, do, dec, 0.7)
    b = OLN.backward_recurrent(t.parent, t.seg_len, q, k, v, do, dec, 0.7)
    for x, y in zip(a, b):
        assert np.abs(x - y).max() <= 1e-10 * max(1.0, np.abs(x).max())


def test_backward_chain_no_decay_equals_torch_autograd():
    """A single chain with gamma = 1 is causal linear attention, scale * tril(Q K^T) V:
    its gradients from torch autograd equal the oracle's backward."""
    t = WT.chain_tree([6, 5])
    q, k, v = rnd(t.n_tokens, 2, 1, 4, 21)
    do = np.random.default_rng(22).normal(size=(t.n_tokens, 2, 4))
    s = 0.45
    dq, dk, dv = OLN.backward_parallel(t.parent, t.seg_len, q, k, v, do, [1.0], s)
    Q = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    K = torch.tensor(k, dtype=torch.float64, requires_grad=True)
    V = torch.tensor(v, dtype=torch.float64, requires_grad=True)
    out = torch.stack([s * torch.tril(Q[:, h] @ K[:, 0].T) @ V[:, 0] for h in range(2)], dim=1)
    (out * torch.tensor(do)).sum().backward()
    for mine, ref in ((dq, Q.grad), (dk, K.grad), (dv, V.grad)):
        assert np.abs(mine - ref.numpy()).max() < 1e-12
