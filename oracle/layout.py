"""Tree bookkeeping for the oracle: packed order, trajectories, ancestor sets.

Packing convention (the data format shared with the library's callers): the
compact token sequence lists node segments in depth-first pre-order, roots in
ascending node id, children of a node in ascending node id.  The pages fix a
depth-first traversal of the tree (AReaL-DTA abstract); the sibling order is
a reading of ours (ascending id).

Everything here walks parent pointers; nothing uses the library's planner.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np


def validate(parent: Sequence[int], seg_len: Sequence[int]) -> None:
    n = len(parent)
    if n == 0 or len(seg_len) != n:
        raise ValueError("empty tree or length mismatch")
    for v in range(n):
        if not (-1 <= parent[v] < n) or parent[v] == v:
            raise ValueError(f"bad parent for node {v}")
        if seg_len[v] <= 0:
            raise ValueError(f"segment length of node {v} must be > 0")
    for v in range(n):          # every node must reach a root
        u, steps = v, 0
        while parent[u] >= 0:
            u = parent[u]
            steps += 1
            if steps > n:
                raise ValueError("cycle in parent pointers")


def children(parent: Sequence[int]) -> List[List[int]]:
    ch: List[List[int]] = [[] for _ in parent]
    for v, p in enumerate(parent):
        if p >= 0:
            ch[p].append(v)
    for c in ch:
        c.sort()
    return ch


def packed_layout(parent: Sequence[int], seg_len: Sequence[int]) -> Tuple[List[int], np.ndarray, int]:
    """(order, node_off, N): DFS pre-order of node ids and each node's first token."""
    validate(parent, seg_len)
    ch = children(parent)
    order: List[int] = []
    for r in sorted(v for v in range(len(parent)) if parent[v] < 0):
        stack = [r]
        while stack:
            u = stack.pop()
            order.append(u)
            stack.extend(reversed(ch[u]))
    node_off = np.zeros(len(parent), dtype=np.int64)
    pos = 0
    for u in order:
        node_off[u] = pos
        pos += seg_len[u]
    return order, node_off, pos


def token_nodes(parent, seg_len) -> np.ndarray:
    """node id of every compact token."""
    order, off, N = packed_layout(parent, seg_len)
    tn = np.empty(N, dtype=np.int64)
    for u in order:
        tn[off[u]:off[u] + seg_len[u]] = u
    return tn


def root_path(parent, v) -> List[int]:
    """Node ids from the root down to v, found by walking parent pointers."""
    path = []
    while v >= 0:
        path.append(v)
        v = parent[v]
    return path[::-1]


def leaves(parent) -> List[int]:
    ch = children(parent)
    return [v for v in range(len(parent)) if not ch[v]]


def trajectories(parent, seg_len) -> List[Tuple[int, np.ndarray]]:
    """[(leaf, compact token indices of its root-to-leaf trajectory)], leaves ascending."""
    _, off, _ = packed_layout(parent, seg_len)
    out = []
    for leaf in leaves(parent):
        idx = np.concatenate([np.arange(off[u], off[u] + seg_len[u]) for u in root_path(parent, leaf)])
        out.append((leaf, idx))
    return out


def multiplicity(parent, seg_len) -> np.ndarray:
    """Per compact token: how many trajectories contain it (leaves under its node)."""
    N = packed_layout(parent, seg_len)[2]
    mult = np.zeros(N, dtype=np.int64)
    for _, idx in trajectories(parent, seg_len):
        mult[idx] += 1
    return mult


def ancestor_matrix(parent) -> np.ndarray:
    """A[w, u] = True iff u is w or an ancestor of w (parent walking)."""
    n = len(parent)
    A = np.zeros((n, n), dtype=bool)
    for w in range(n):
        for u in root_path(parent, w):
            A[w, u] = True
    return A


def mask_rows(parent, seg_len, rows: np.ndarray, tn: np.ndarray = None, A: np.ndarray = None) -> np.ndarray:
    """Dense attention mask for the given query rows: mask[r, j] is True iff
    key j lies on row r's root-to-node path and, inside row r's own segment,
    j <= r (causal).  Built from ancestor sets, not from the library's plan."""
    if tn is None:
        tn = token_nodes(parent, seg_len)
    if A is None:
        A = ancestor_matrix(parent)
    rows = np.asarray(rows, dtype=np.int64)
    N = tn.shape[0]
    cols = np.arange(N)
    wn = tn[rows]
    m = A[wn][:, tn]
    same = wn[:, None] == tn[None, :]
    m &= ~same | (cols[None, :] <= rows[:, None])
    return m


def dense_mask(parent, seg_len) -> np.ndarray:
    N = packed_layout(parent, seg_len)[2]
    return mask_rows(parent, seg_len, np.arange(N))
