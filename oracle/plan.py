"""Brute-force tile plan from the dense ancestor mask (test infrastructure).

The planner the library ships derives everything from one per-token number
(the end of the token's subtree in packed order).  This module derives the
same quantities the slow way, from the definition: the dense mask of which key
each query attends to (built by walking parent pointers), so that the two can
be compared bit for bit.

Quantities (tile size B for both queries and keys, N compact tokens,
T = ceil(N / B) tiles):

* ``node_order`` / ``node_off`` -- the packed layout (DFS pre-order).
* ``subend[j]`` -- one past the last query that attends to key j.  The test
  suite also checks, here, that the queries of key j are exactly [j, subend[j]).
* ``intervals[t]`` -- the maximal runs of key indices attended to by any
  query row of q-tile t, sorted, half-open [lo, hi).
* ``tiles[t]`` -- (kv-tile c, class) for every kv-tile with at least one
  attended pair in the (t, c) block, ascending c; class FULL when every valid
  (query, key) pair in the block is attended, PARTIAL otherwise.  Pairs with an
  index >= N are not valid and are ignored.
* ``kv_range[c]`` -- half-open range of q-tiles with a non-empty (t, c) block.

The plan lists key intervals and full / partial / empty tiles per query tile:
the AReaL-DTA abstract faults packed tree-mask methods for poor scaling, and
skipping empty tiles removes the quadratic mask scan.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np

from . import layout

FULL = 1
PARTIAL = 2


def _runs(cols: np.ndarray):
    """Maximal runs of True in a boolean vector as half-open intervals."""
    x = np.concatenate([[False], cols, [False]]).astype(np.int8)
    dx = np.diff(x)
    starts = np.nonzero(dx == 1)[0]
    ends = np.nonzero(dx == -1)[0]
    return list(zip(starts.tolist(), ends.tolist()))


def brute_plan(parent, seg_len, block: int = 128, qtiles: Optional[Sequence[int]] = None) -> Dict:
    """Plan quantities from the dense mask.  ``qtiles`` restricts the per-tile
    outputs (intervals, tiles) to a sample of q-tiles for large trees."""
    order, off, N = layout.packed_layout(parent, seg_len)
    tn = layout.token_nodes(parent, seg_len)
    A = layout.ancestor_matrix(parent)
    T = (N + block - 1) // block
    all_tiles = qtiles is None
    qtiles = range(T) if qtiles is None else list(qtiles)
    intervals: Dict[int, List] = {}
    tiles: Dict[int, List] = {}
    kv_lo = np.full(T, T, dtype=np.int64)
    kv_hi = np.zeros(T, dtype=np.int64)
    # subend by definition: last attending query + 1 (exact for every key only
    # when all q-tiles are visited)
    subend = np.zeros(N, dtype=np.int64)
    contiguous = True
    for t in qtiles:
        a, b = t * block, min(N, (t + 1) * block)
        M = layout.mask_rows(parent, seg_len, np.arange(a, b), tn, A)      # [rows, N]
        cols = M.any(axis=0)
        intervals[t] = _runs(cols)
        lst = []
        for c in range(T):
            c0, c1 = c * block, min(N, (c + 1) * block)
            blk = M[:, c0:c1]
            cnt = int(blk.sum())
            if cnt == 0:
                continue
            lst.append((c, FULL if cnt == blk.size else PARTIAL))
            kv_lo[c] = min(kv_lo[c], t)
            kv_hi[c] = max(kv_hi[c], t + 1)
        tiles[t] = lst
        if all_tiles:
            rows_any = np.nonzero(M.any(axis=0))[0]
            for j in rows_any:
                last = a + int(np.nonzero(M[:, j])[0].max()) + 1
                subend[j] = max(subend[j], last)
    out = {"N": N, "T": T, "node_order": order, "node_off": off, "intervals": intervals,
           "tiles": tiles}
    if all_tiles:
        out["subend"] = subend
        out["kv_range"] = list(zip(kv_lo.tolist(), kv_hi.tolist()))
    return out


def key_query_sets_contiguous(parent, seg_len) -> bool:
    """True iff, for every key j, the attending queries are exactly
    [j, max attending query] (checked on the dense mask; small N only)."""
    M = layout.dense_mask(parent, seg_len)
    N = M.shape[0]
    for j in range(N):
        rows = np.nonzero(M[:, j])[0]
        if rows.size == 0 or rows[0] != j or rows[-1] - rows[0] + 1 != rows.size:
            return False
    return True


def pair_count(parent, seg_len) -> int:
    """Number of attended (query, key) pairs, by walking each token's path."""
    order, off, N = layout.packed_layout(parent, seg_len)
    total = 0
    for u in range(len(parent)):
        anc = sum(seg_len[w] for w in layout.root_path(parent, u)[:-1])
        L = seg_len[u]
        total += L * anc + L * (L + 1) // 2
    return total
