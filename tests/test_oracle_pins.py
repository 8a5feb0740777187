"""Pins for the fp64 oracle against things other than itself (CPU only).

* single chain == torch scaled_dot_product_attention(is_causal=True), forward
  and, through autograd, backward;
* per-trajectory SDPA + autograd on random trees (the equivalence the
  AReaL-DTA and HARTS abstracts require, computed by a library routine);
* pure-Python brute force on every small rooted tree;
* closed forms at constant logits;
* central finite differences of <O, dO>;
* the second (compact, masked) formula;
* invariants: dO split, sibling permutation, chain merge, forest, star.
"""
import itertools
import math

import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import layout as OL
from workloads import trees as WT

F64 = torch.float64


def rand_inputs(N, hq, hkv, d, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(N, hq, d, generator=g, dtype=F64) * std
    k = torch.randn(N, hkv, d, generator=g, dtype=F64) * std
    v = torch.randn(N, hkv, d, generator=g, dtype=F64)
    do = torch.randn(N, hq, d, generator=g, dtype=F64)
    return q, k, v, do


def sdpa(q, k, v, scale):
    """q [L, hq, d], k/v [L, hkv, d] -> O [L, hq, d] via torch SDPA (causal)."""
    g = q.shape[1] // k.shape[1]
    kk = k.repeat_interleave(g, dim=1)
    vv = v.repeat_interleave(g, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(
        q.transpose(0, 1)[None], kk.transpose(0, 1)[None], vv.transpose(0, 1)[None],
        is_causal=True, scale=scale)
    return o[0].transpose(0, 1)


# ---------------------------------------------------------------------------
# single chain == SDPA
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("lens,hq,hkv,d,scale", [([7], 2, 2, 8, 0.35), ([5, 3, 9], 4, 2, 16, 0.25),
                                                  ([1, 1, 1, 4], 6, 3, 4, 1.0)])
def test_chain_equals_sdpa(lens, hq, hkv, d, scale):
    t = WT.chain_tree(lens)
    N = t.n_tokens
    q, k, v, do = rand_inputs(N, hq, hkv, d, seed=11)
    O, lse = OA.forward(t.parent, t.seg_len, q, k, v, scale)
    qr, kr, vr = (x.clone().requires_grad_(True) for x in (q, k, v))
    o_ref = sdpa(qr, kr, vr, scale)
    np.testing.assert_allclose(O, o_ref.detach().numpy(), atol=1e-12, rtol=0)
    (o_ref * do).sum().backward()
    dq, dk, dv = OA.backward(t.parent, t.seg_len, q, k, v, do, scale)
    np.testing.assert_allclose(dq, qr.grad.numpy(), atol=1e-11, rtol=0)
    np.testing.assert_allclose(dk, kr.grad.numpy(), atol=1e-11, rtol=0)
    np.testing.assert_allclose(dv, vr.grad.numpy(), atol=1e-11, rtol=0)
    # LSE: softmax rows built from it must sum to one (scipy logsumexp of the same logits too)
    from scipy.special import logsumexp
    g = hq // hkv
    for h in range(hq):
        s = scale * (q[:, h, :] @ k[:, h // g, :].T).numpy()
        s = np.where(np.tril(np.ones((N, N), dtype=bool)), s, -np.inf)
        np.testing.assert_allclose(lse[h], logsumexp(s, axis=1), atol=1e-12)
        np.testing.assert_allclose(np.exp(s - lse[h][:, None]).sum(axis=1), 1.0, atol=1e-12)


# ---------------------------------------------------------------------------
# trajectory-wise SDPA + autograd on random trees
# ---------------------------------------------------------------------------

def trajectory_sdpa_reference(t, q, k, v, do, scale, assign="first"):
    """Library computation of the required equivalence: each trajectory runs
    SDPA on its own; the compact output takes the first copy (or the mean of
    the copies); autograd of <O_compact, dO> gives the compact gradients."""
    qr, kr, vr = (x.clone().requires_grad_(True) for x in (q, k, v))
    N = q.shape[0]
    trajs = OL.trajectories(t.parent, t.seg_len)
    mult = torch.zeros(N, dtype=F64)
    for _, idx in trajs:
        mult[torch.as_tensor(idx)] += 1
    acc = torch.zeros_like(q)
    seen = torch.zeros(N, dtype=torch.bool)
    for _, idx in trajs:
        ii = torch.as_tensor(idx)
        o = sdpa(qr[ii], kr[ii], vr[ii], scale)
        if assign == "first":
            keep = (~seen[ii]).to(F64)[:, None, None]
            seen[ii] = True
            acc = acc.index_add(0, ii, o * keep)
        else:
            acc = acc.index_add(0, ii, o / mult[ii][:, None, None])
    (acc * do).sum().backward()
    return acc.detach().numpy(), qr.grad.numpy(), kr.grad.numpy(), vr.grad.numpy()


@pytest.mark.parametrize("seed", range(6))
def test_random_trees_match_trajectory_sdpa(seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(1, 9))
    t = WT.random_tree(rng, n, [1, 2, 3, 5, 8, 13], n_roots=1 + (seed % 2))
    hq, hkv = [(2, 2), (4, 2), (6, 3)][seed % 3]
    q, k, v, do = rand_inputs(t.n_tokens, hq, hkv, 8, seed=seed)
    scale = 0.4
    O, _ = OA.forward(t.parent, t.seg_len, q, k, v, scale)
    dq, dk, dv = OA.backward(t.parent, t.seg_len, q, k, v, do, scale)
    for assign in ("first", "mean"):
        o_ref, gq, gk, gv = trajectory_sdpa_reference(t, q, k, v, do, scale, assign)
        np.testing.assert_allclose(O, o_ref, atol=1e-12, rtol=0)
        np.testing.assert_allclose(dq, gq, atol=1e-11, rtol=0)
        np.testing.assert_allclose(dk, gk, atol=1e-11, rtol=0)
        np.testing.assert_allclose(dv, gv, atol=1e-11, rtol=0)


# ---------------------------------------------------------------------------
# brute force, pure Python, every rooted tree of <= 4 nodes (+ samples of 5)
# ---------------------------------------------------------------------------

def all_rooted_trees(n):
    for par in itertools.product(range(-1, n), repeat=n):
        if sum(1 for p in par if p < 0) != 1:
            continue
        if any(par[v] == v for v in range(n)):
            continue
        ok = True
        for v in range(n):
            u, s = v, 0
            while par[u] >= 0:
                u = par[u]
                s += 1
                if s > n:
                    ok = False
                    break
            if not ok:
                break
        if ok:
            yield list(par)


def brute_offsets(parent, seg_len):
    """Packed layout by plain recursion (roots, then children, ascending id)."""
    n = len(parent)
    off = [0] * n
    pos = [0]

    def visit(u):
        off[u] = pos[0]
        pos[0] += seg_len[u]
        for c in range(n):
            if parent[c] == u:
                visit(c)
    for r in range(n):
        if parent[r] < 0:
            visit(r)
    return off, pos[0]


def brute_forward(parent, seg_len, q, k, v, scale):
    """Loops only: each token's softmax over its own root-to-node path."""
    off, N = brute_offsets(parent, seg_len)
    hq, hkv, d = q.shape[1], k.shape[1], q.shape[2]
    g = hq // hkv
    O = [[[0.0] * d for _ in range(hq)] for _ in range(N)]
    LSE = [[0.0] * N for _ in range(hq)]
    for w in range(len(parent)):
        chain = []
        u = w
        while u >= 0:
            chain.append(u)
            u = parent[u]
        chain.reverse()
        for p in range(seg_len[w]):
            i = off[w] + p
            keys = []
            for u in chain[:-1]:
                keys += list(range(off[u], off[u] + seg_len[u]))
            keys += list(range(off[w], i + 1))
            for h in range(hq):
                s = [scale * sum(float(q[i, h, x]) * float(k[j, h // g, x]) for x in range(d)) for j in keys]
                m = max(s)
                e = [math.exp(z - m) for z in s]
                tot = sum(e)
                LSE[h][i] = m + math.log(tot)
                for x in range(d):
                    O[i][h][x] = sum(e[a] * float(v[j, h // g, x]) for a, j in enumerate(keys)) / tot
    return np.array(O), np.array(LSE)


def small_cases():
    rng = np.random.default_rng(7)
    cases = []
    for n in range(1, 5):
        for par in all_rooted_trees(n):
            cases.append((par, [int(x) for x in rng.choice([1, 2, 3], size=n)]))
    five = list(all_rooted_trees(5))
    for i in rng.choice(len(five), size=25, replace=False):
        cases.append((five[int(i)], [int(x) for x in rng.choice([1, 2, 3], size=5)]))
    return cases


def test_brute_force_small_trees():
    cases = small_cases()
    assert len(cases) >= 1 + 2 + 9 + 64 + 25
    for ci, (par, lens) in enumerate(cases):
        N = sum(lens)
        q, k, v, do = rand_inputs(N, 2, 1, 4, seed=ci)
        O, lse = OA.forward(par, lens, q, k, v, 0.7)
        Ob, lseb = brute_forward(par, lens, q, k, v, 0.7)
        np.testing.assert_allclose(O, Ob, atol=1e-12, rtol=0)
        np.testing.assert_allclose(lse, lseb, atol=1e-12, rtol=0)
        Om, lsem = OA.masked_forward(par, lens, q, k, v, 0.7)
        np.testing.assert_allclose(Om, Ob, atol=1e-12, rtol=0)
        np.testing.assert_allclose(lsem, lseb, atol=1e-12, rtol=0)


def test_brute_offsets_match_layout():
    for par, lens in small_cases():
        off, N = brute_offsets(par, lens)
        order, off2, N2 = OL.packed_layout(par, lens)
        assert N == N2 and list(off) == list(off2)


# ---------------------------------------------------------------------------
# closed forms at constant logits (q = 0): uniform attention over the path
# ---------------------------------------------------------------------------

def test_closed_form_uniform_attention():
    t = WT.tiny_binary_tree()
    t = WT.Tree("small_binary", t.parent, [4, 2, 3, 1, 2, 3, 2])
    N = t.n_tokens
    _, k, v, do = rand_inputs(N, 2, 2, 4, seed=3)
    q = torch.zeros(N, 2, 4, dtype=F64)
    O, lse = OA.forward(t.parent, t.seg_len, q, k, v, 1.0)
    dq, dk, dv = OA.backward(t.parent, t.seg_len, q, k, v, do, 1.0)
    # by hand: token i attends to count(i) keys = tokens on the path up to i
    off, _ = brute_offsets(t.parent, t.seg_len)
    keysets = {}
    for w in range(t.n_nodes):
        path = []
        u = w
        while u >= 0:
            path.append(u)
            u = t.parent[u]
        prefix = [j for u in reversed(path[1:]) for j in range(off[u], off[u] + t.seg_len[u])]
        for p in range(t.seg_len[w]):
            i = off[w] + p
            keysets[i] = prefix + list(range(off[w], i + 1))
    vv = v.numpy()
    dd = do.numpy()
    dv_ref = np.zeros_like(vv)
    for i, ks in keysets.items():
        np.testing.assert_allclose(lse[:, i], math.log(len(ks)), atol=1e-13)
        np.testing.assert_allclose(O[i], vv[ks].mean(axis=0), atol=1e-13)
        for j in ks:
            dv_ref[j] += dd[i] / len(ks)
    np.testing.assert_allclose(dv, dv_ref, atol=1e-13)
    np.testing.assert_allclose(dk, 0.0, atol=1e-13)      # dK = scale * dS^T Q with Q = 0


# ---------------------------------------------------------------------------
# finite differences of L = <O, dO>
# ---------------------------------------------------------------------------

def test_finite_differences():
    t = WT.Tree("fd", [-1, 0, 0, 1], [2, 2, 1, 2])
    N = t.n_tokens
    q, k, v, do = rand_inputs(N, 2, 1, 3, seed=5)
    scale = 0.8
    dq, dk, dv = OA.backward(t.parent, t.seg_len, q, k, v, do, scale)
    dd = do.numpy()

    def loss(qq, kk, vvv):
        O, _ = OA.forward(t.parent, t.seg_len, qq, kk, vvv, scale)
        return float((O * dd).sum())

    h = 1e-6
    for name, base, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros(base.shape)
        arr = base.numpy()
        for idx in np.ndindex(*arr.shape):
            xp = arr.copy()
            xm = arr.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q.numpy(), "k": k.numpy(), "v": v.numpy()}
            args_m = dict(args_p)
            args_p[name] = xp
            args_m[name] = xm
            fd[idx] = (loss(args_p["q"], args_p["k"], args_p["v"]) -
                       loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
        rel = np.linalg.norm(fd - grad) / np.linalg.norm(grad)
        assert rel < 1e-6, (name, rel)


# ---------------------------------------------------------------------------
# second formula and invariants
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(4))
def test_masked_formula_agrees(seed):
    rng = np.random.default_rng(200 + seed)
    t = WT.random_tree(rng, int(rng.integers(2, 12)), [1, 3, 7, 16, 40], n_roots=1 + seed % 3)
    q, k, v, do = rand_inputs(t.n_tokens, 4, 2, 8, seed=seed)
    a = OA.forward(t.parent, t.seg_len, q, k, v, 0.3)
    b = OA.masked_forward(t.parent, t.seg_len, q, k, v, 0.3)
    np.testing.assert_allclose(a[0], b[0], atol=1e-12)
    np.testing.assert_allclose(a[1], b[1], atol=1e-12)
    ga = OA.backward(t.parent, t.seg_len, q, k, v, do, 0.3)
    gb = OA.masked_backward(t.parent, t.seg_len, q, k, v, do, 0.3)
    gc = OA.backward(t.parent, t.seg_len, q, k, v, do, 0.3, split="first")
    for x, y, z in zip(ga, gb, gc):
        np.testing.assert_allclose(x, y, atol=1e-11)
        np.testing.assert_allclose(x, z, atol=1e-10)


def per_node(t, arr):
    """{node: rows of a compact [N, ...] array} using the packed layout."""
    _, off, _ = OL.packed_layout(t.parent, t.seg_len)
    return {u: arr[off[u]:off[u] + t.seg_len[u]] for u in range(t.n_nodes)}


def test_sibling_permutation_invariance():
    rng = np.random.default_rng(9)
    t = WT.random_tree(rng, 9, [2, 3, 5], n_roots=1)
    perm = rng.permutation(t.n_nodes)                       # relabel: old -> new id
    inv = np.argsort(perm)
    t2 = WT.Tree("perm", [-1] * t.n_nodes, [0] * t.n_nodes)
    for old in range(t.n_nodes):
        p = t.parent[old]
        t2.parent[perm[old]] = -1 if p < 0 else int(perm[p])
        t2.seg_len[perm[old]] = t.seg_len[old]
    # draw per-node values and pack them in each tree's own order
    q, k, v, do = rand_inputs(t.n_tokens, 2, 1, 4, seed=1)
    _, off1, _ = OL.packed_layout(t.parent, t.seg_len)
    _, off2, _ = OL.packed_layout(t2.parent, t2.seg_len)
    idx = np.concatenate([np.arange(off1[inv[u2]], off1[inv[u2]] + t2.seg_len[u2])
                          for u2 in OL.packed_layout(t2.parent, t2.seg_len)[0]])
    ii = torch.as_tensor(idx)
    o1, l1 = OA.forward(t.parent, t.seg_len, q, k, v, 0.5)
    o2, l2 = OA.forward(t2.parent, t2.seg_len, q[ii], k[ii], v[ii], 0.5)
    np.testing.assert_allclose(o1[idx], o2, atol=1e-12)
    np.testing.assert_allclose(l1[:, idx], l2, atol=1e-12)
    g1 = OA.backward(t.parent, t.seg_len, q, k, v, do, 0.5)
    g2 = OA.backward(t2.parent, t2.seg_len, q[ii], k[ii], v[ii], do[ii], 0.5)
    for a, b in zip(g1, g2):
        np.testing.assert_allclose(a[idx], b, atol=1e-12)


def test_chain_merge_and_star_and_forest():
    q, k, v, do = rand_inputs(12, 2, 2, 4, seed=2)
    chain = WT.chain_tree([3, 4, 5])
    merged = WT.Tree("merged", [-1], [12])
    star1 = WT.Tree("star1", [-1, 0], [7, 5])
    outs = [OA.forward(t.parent, t.seg_len, q, k, v, 0.6) for t in (chain, merged, star1)]
    grads = [OA.backward(t.parent, t.seg_len, q, k, v, do, 0.6) for t in (chain, merged, star1)]
    for o in outs[1:]:
        np.testing.assert_allclose(o[0], outs[0][0], atol=1e-12)
        np.testing.assert_allclose(o[1], outs[0][1], atol=1e-12)
    for g in grads[1:]:
        for a, b in zip(g, grads[0]):
            np.testing.assert_allclose(a, b, atol=1e-12)
    # forest of two trees == each tree alone
    forest = WT.Tree("forest", [-1, 0, -1, 2, 2], [3, 2, 2, 3, 2])
    qf, kf, vf, dof = rand_inputs(12, 2, 1, 4, seed=4)
    of, lf = OA.forward(forest.parent, forest.seg_len, qf, kf, vf, 0.6)
    gf = OA.backward(forest.parent, forest.seg_len, qf, kf, vf, dof, 0.6)
    a, b = slice(0, 5), slice(5, 12)
    oa, la = OA.forward([-1, 0], [3, 2], qf[a], kf[a], vf[a], 0.6)
    ob, lb = OA.forward([-1, 0, 0], [2, 3, 2], qf[b], kf[b], vf[b], 0.6)
    np.testing.assert_allclose(of[a], oa, atol=1e-12)
    np.testing.assert_allclose(of[b], ob, atol=1e-12)
    ga = OA.backward([-1, 0], [3, 2], qf[a], kf[a], vf[a], dof[a], 0.6)
    gb = OA.backward([-1, 0, 0], [2, 3, 2], qf[b], kf[b], vf[b], dof[b], 0.6)
    for x, y, z in zip(gf, ga, gb):
        np.testing.assert_allclose(x[a], y, atol=1e-12)
        np.testing.assert_allclose(x[b], z, atol=1e-12)


def test_copies_agree_and_rows_sum_to_one():
    t = WT.tiny_binary_tree()
    t = WT.Tree("b", t.parent, [8, 4, 4, 4, 4, 4, 4])
    q, k, v, _ = rand_inputs(t.n_tokens, 2, 2, 4, seed=8)
    info = {}
    O, lse = OA.forward(t.parent, t.seg_len, q, k, v, 1.3, info=info)
    assert info["copy_disagreement"] < 1e-12
    M = OL.dense_mask(t.parent, t.seg_len)
    for h in range(2):
        s = 1.3 * (q[:, h, :] @ k[:, h, :].T).numpy()
        p = np.where(M, np.exp(s - lse[h][:, None]), 0.0)
        np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)


def test_sampled_rows_and_keys_match_full():
    rng = np.random.default_rng(31)
    t = WT.random_tree(rng, 7, [3, 6, 11], n_roots=1)
    q, k, v, do = rand_inputs(t.n_tokens, 4, 2, 8, seed=6)
    O, lse = OA.forward(t.parent, t.seg_len, q, k, v, 0.45)
    dq, dk, dv = OA.backward(t.parent, t.seg_len, q, k, v, do, 0.45)
    rows = rng.choice(t.n_tokens, size=9, replace=False)
    Or, lr = OA.forward_rows(t.parent, t.seg_len, q, k, v, 0.45, rows)
    np.testing.assert_allclose(Or, O[rows], atol=1e-12)
    np.testing.assert_allclose(lr, lse[:, rows], atol=1e-12)
    dqr = OA.backward_rows_dq(t.parent, t.seg_len, q, k, v, do, 0.45, rows)
    np.testing.assert_allclose(dqr, dq[rows], atol=1e-12)
    dkr, dvr = OA.backward_keys_dkdv(t.parent, t.seg_len, q, k, v, do, 0.45, rows)
    np.testing.assert_allclose(dkr, dk[rows], atol=1e-12)
    np.testing.assert_allclose(dvr, dv[rows], atol=1e-12)
