"""Loss-boundary quantities, the slow and obvious way (test infrastructure).

Everything starts from the expanded trajectories (one per leaf, leaves in
ascending node id, tokens of the root-to-leaf path in order), found by walking
parent pointers; fp64 throughout.

* position id of a compact token: its index in any trajectory containing it;
* multiplicity: the number of trajectories containing it (``layout``);
* next-token log-probs of trajectory l: log_softmax(logits[row of position p])
  at the token id of position p + 1, for p = 0 .. len - 2 (HARTS abstract: a
  compact token stands for the trajectory tokens it replaces; restoring the
  per-trajectory log-probs is the step that precedes the loss);
* subtree advantages (TreePO: advantages over sub-trees from collective
  descendant outcomes; simple vs size-weighted subgroup aggregation; the root
  group optional).  Our reading, written out in the library header:
  subgroups of leaf l = nodes u on its root path with at least two leaves below;
  a_u(l) = R_l - mean_u, optionally / (std_u + eps) (population std); A(l) the
  plain or |G(u)|-weighted mean of a_u(l); node coefficient = sum of A over the
  node's leaves; token coefficient = its node's coefficient.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np

from . import layout


def position_ids(parent, seg_len) -> np.ndarray:
    N = layout.packed_layout(parent, seg_len)[2]
    pos = np.full(N, -1, dtype=np.int64)
    for _, idx in layout.trajectories(parent, seg_len):
        for p, t in enumerate(idx):
            if pos[t] >= 0 and pos[t] != p:
                raise AssertionError("a token at two positions")
            pos[t] = p
    return pos


def row_logsumexp(logits: np.ndarray) -> np.ndarray:
    x = np.asarray(logits, dtype=np.float64)
    m = x.max(axis=1)
    return m + np.log(np.exp(x - m[:, None]).sum(axis=1))


def traj_logprobs(parent, seg_len, logits, tokens, rows_lse=None) -> np.ndarray:
    """Concatenated next-token log-probs of every trajectory (leaves ascending)."""
    x = np.asarray(logits, dtype=np.float64)
    lse = row_logsumexp(x) if rows_lse is None else rows_lse
    tok = np.asarray(tokens)
    out: List[float] = []
    for _, idx in layout.trajectories(parent, seg_len):
        for p in range(len(idx) - 1):
            r, s = idx[p], idx[p + 1]
            out.append(x[r, tok[s]] - lse[r])
    return np.asarray(out, dtype=np.float64)


def scale_rows(x, w) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    return x * np.asarray(w, dtype=np.float64).reshape((-1,) + (1,) * (x.ndim - 1))


def subtree_advantage(parent, seg_len, rewards, norm_std=False, size_weighted=False, no_root=False,
                      eps=1e-6) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """(A per leaf ascending id, coefficient per node id, coefficient per compact token)."""
    leaves = layout.leaves(parent)
    R = {leaf: float(r) for leaf, r in zip(leaves, rewards)}
    below = {u: [] for u in range(len(parent))}           # leaves under each node
    for leaf in leaves:
        for u in layout.root_path(parent, leaf):
            below[u].append(leaf)
    A = {}
    for leaf in leaves:
        num = den = 0.0
        for u in layout.root_path(parent, leaf):
            g = below[u]
            if len(g) < 2 or (no_root and parent[u] < 0):
                continue
            vals = [R[x] for x in g]
            mean = sum(vals) / len(vals)
            a = R[leaf] - mean
            if norm_std:
                std = (sum((v - mean) ** 2 for v in vals) / len(vals)) ** 0.5
                a /= std + eps
            wgt = float(len(g)) if size_weighted else 1.0
            num += wgt * a
            den += wgt
        A[leaf] = num / den if den > 0 else 0.0
    node_c = np.array([sum(A[x] for x in below[u]) for u in range(len(parent))], dtype=np.float64)
    tn = layout.token_nodes(parent, seg_len)
    return np.array([A[x] for x in leaves], dtype=np.float64), node_c, node_c[tn]
