"""Batching many rollout trees (``include/tree_batch.h``): per-tree
ancestor-pair work, LPT assignment to data-parallel replicas, token-capped
microbatches, and the packed forest of a group of trees.  Host only; the work
runs in the C++ library, this module marshals arguments.

    batch = TreeBatch([(parent, seg_len), ...])   # parent indices local to each tree
    pairs, tokens = batch.work()
    replica_of, load = batch_assign(pairs, n_replicas)
    mb_of, n_mb = batch_microbatches(pairs, tokens, replica_of, replica=0, max_tokens=65536)
    parent, seg_len, tree_of = batch.forest(mb_of == 0)   # one plan per microbatch
"""
from __future__ import annotations

import ctypes as C
from typing import Sequence, Tuple

import numpy as np

from . import _binding as B


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def _p32(a):
    return a.ctypes.data_as(B.c_int32_p)


def _p64(a):
    return a.ctypes.data_as(B.c_int64_p)


def _concat(trees: Sequence[Tuple[Sequence[int], Sequence[int]]]):
    sizes = [len(p) for p, _ in trees]
    ptr = _i32(np.concatenate([[0], np.cumsum(sizes, dtype=np.int64)]) if trees else [0])
    parent = _i32(np.concatenate([np.asarray(p, dtype=np.int32) for p, _ in trees]) if trees else [])
    seg = _i32(np.concatenate([np.asarray(s, dtype=np.int32) for _, s in trees]) if trees else [])
    for (p, s) in trees:
        if len(p) != len(s):
            raise ValueError("parent and seg_len differ in length")
    return ptr, parent, seg


class TreeBatch:
    """Many trees concatenated once for repeated batching calls."""

    def __init__(self, trees):
        self.n = len(trees)
        self.ptr, self.parent, self.seg = _concat(trees)

    def work(self) -> Tuple[np.ndarray, np.ndarray]:
        """(ancestor pairs, compact tokens) of each tree."""
        pairs, tokens = np.zeros(self.n, np.int64), np.zeros(self.n, np.int64)
        B.check(B.load().tree_attn_batch_work(self.n, _p32(self.ptr), _p32(self.parent), _p32(self.seg),
                                              _p64(pairs), _p64(tokens)), "tree_attn_batch_work")
        return pairs, tokens

    def forest(self, select) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
        """The forest of the selected trees: (parent, seg_len, source tree of each node)."""
        sel = np.ascontiguousarray(np.asarray(select, dtype=bool).astype(np.uint8))
        if len(sel) != self.n:
            raise ValueError("select needs one flag per tree")
        sizes = np.diff(self.ptr)
        total = int(sizes[sel.astype(bool)].sum()) if self.n else 0
        op, os_, ot = (np.zeros(max(total, 1), np.int32) for _ in range(3))
        k = C.c_int32(0)
        B.check(B.load().tree_attn_batch_forest(self.n, _p32(self.ptr), _p32(self.parent), _p32(self.seg),
                                                sel.ctypes.data_as(B.c_uint8_p), _p32(op), _p32(os_), _p32(ot),
                                                C.byref(k)), "tree_attn_batch_forest")
        m = int(k.value)
        return op[:m], os_[:m], ot[:m]


def batch_work(trees) -> Tuple[np.ndarray, np.ndarray]:
    """(ancestor pairs, compact tokens) of each tree."""
    return TreeBatch(trees).work()


def batch_assign(work, n_replicas: int) -> Tuple[np.ndarray, np.ndarray]:
    """LPT: (replica of each tree, summed work of each replica)."""
    lib = B.load()
    w = _i64(work)
    rep = np.zeros(len(w), np.int32)
    load = np.zeros(max(n_replicas, 0), np.int64)
    B.check(lib.tree_attn_batch_assign(len(w), _p64(w), n_replicas, _p32(rep), _p64(load)),
            "tree_attn_batch_assign")
    return rep, load


def batch_microbatches(work, tokens, replica_of, replica: int, max_tokens: int) -> Tuple[np.ndarray, int]:
    """First-fit microbatches of one replica's trees: (microbatch of each tree or -1, count)."""
    lib = B.load()
    w, t, r = _i64(work), _i64(tokens), _i32(replica_of)
    mb = np.zeros(len(w), np.int32)
    cnt = C.c_int32(0)
    B.check(lib.tree_attn_batch_microbatches(len(w), _p64(w), _p64(t), _p32(r), replica, max_tokens, _p32(mb),
                                             C.byref(cnt)), "tree_attn_batch_microbatches")
    return mb, int(cnt.value)


def batch_forest(trees, select) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """The forest of the selected trees: (parent, seg_len, source tree of each node)."""
    return TreeBatch(trees).forest(select)
