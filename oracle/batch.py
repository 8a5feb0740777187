"""Batching many trees, the slow and obvious way (test infrastructure).

Follows the definitions the batching calls state (AReaL-DTA abstract: trees
assigned to GPUs to balance work; HARTS abstract: microbatches and replica
assignments planned from compact-token work), with these readings of ours:

* work of a tree = its ancestor pairs: the number of (query, key) token pairs
  with the key on the query's root-to-node path (inside the query's own segment:
  key at or before the query).  Counted here by walking parent pointers token by
  token, with no formula;
* replicas by LPT: trees in descending work (ties: ascending index), each onto
  the replica with the least work so far (ties: lowest replica index);
* microbatches of one replica: its trees in the same order, first fit under a
  compact-token cap (a tree above the cap alone);
* the forest of a set of trees: concatenated in ascending tree index, parent
  indices shifted by the nodes before them.

Pure Python loops; sizes in the tests are small.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

from . import layout


def pairs_by_walking(parent: Sequence[int], seg_len: Sequence[int]) -> int:
    """Count attended (query, key) pairs token by token."""
    layout.validate(parent, seg_len)
    total = 0
    for w in range(len(parent)):
        for q in range(seg_len[w]):          # query = token q of node w
            total += q + 1                    # keys of w at or before it
            u = parent[w]
            while u >= 0:                     # every token of every ancestor
                total += seg_len[u]
                u = parent[u]
    return total


def tokens(seg_len: Sequence[int]) -> int:
    return int(sum(seg_len))


def lpt(work: Sequence[int], n_replicas: int) -> Tuple[List[int], List[int]]:
    order = sorted(range(len(work)), key=lambda k: (-work[k], k))
    load = [0] * n_replicas
    rep = [0] * len(work)
    for k in order:
        best = min(range(n_replicas), key=lambda r: (load[r], r))
        rep[k] = best
        load[best] += work[k]
    return rep, load


def microbatches(work: Sequence[int], toks: Sequence[int], replica_of: Sequence[int], replica: int,
                 max_tokens: int) -> Tuple[List[int], int]:
    order = sorted(range(len(work)), key=lambda k: (-work[k], k))
    fill: List[int] = []
    mb = [-1] * len(work)
    for k in order:
        if replica_of[k] != replica:
            continue
        m = 0
        while m < len(fill) and fill[m] + toks[k] > max_tokens:
            m += 1
        if m == len(fill):
            fill.append(0)
        fill[m] += toks[k]
        mb[k] = m
    return mb, len(fill)


def forest(trees, select) -> Tuple[List[int], List[int], List[int]]:
    par: List[int] = []
    seg: List[int] = []
    src: List[int] = []
    for k, ((p, s), on) in enumerate(zip(trees, select)):
        if not on:
            continue
        base = len(par)
        par += [-1 if x < 0 else x + base for x in p]
        seg += list(s)
        src += [k] * len(p)
    return par, seg, src
