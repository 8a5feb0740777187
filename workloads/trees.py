"""Rollout prefix trees shaped like the workloads on the pages.

A tree (or forest) is two arrays over nodes: ``parent[v]`` (-1 for a root)
and ``seg_len[v]`` (tokens in node v's segment, > 0).  Every node is one
segment of shared tokens; a root-to-leaf path is one trajectory.

Shapes and their sources:

* tiny binary tree -- a 64-token prompt, binary branching over two levels of
  32-token segments (4 leaves).  Binary branching is the TreePO tree setting
  (TreePO page, section 3 "Tree Setting").
* GRPO star -- one shared prompt with many sibling responses: the GRPO group
  that TreePO starts from (TreePO page, section 2 "Policy Optimization").
* segment tree -- fixed-length segments, binary branching, early stop and
  fallback until the target width is reached (TreePO page, section 2
  "Segment-level Tree Sampling", "Branching and Fallback"; section 3 "Tree
  Setting": width 16).
* agentic tree -- an irregular multi-turn tree with shared histories
  (HARTS abstract: "irregular rollout trees with shared histories").
* long shared context -- one long shared prefix with many branches
  (AReaL-DTA abstract: rollouts "frequently share long token prefixes").

Trees drawn from a seeded ``numpy.random.default_rng`` are frozen as JSON
under ``workloads/trees/`` by ``make_trees.py`` so that every machine sees the
same shapes whatever its numpy version.
"""
from __future__ import annotations

import dataclasses
import json
import math
import os
from typing import List

import numpy as np

TREE_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "trees")


@dataclasses.dataclass
class Tree:
    name: str
    parent: List[int]
    seg_len: List[int]

    @property
    def n_nodes(self) -> int:
        return len(self.parent)

    @property
    def n_tokens(self) -> int:
        return int(sum(self.seg_len))

    def children(self) -> List[List[int]]:
        ch: List[List[int]] = [[] for _ in self.parent]
        for v, p in enumerate(self.parent):
            if p >= 0:
                ch[p].append(v)
        return ch

    def leaves(self) -> List[int]:
        ch = self.children()
        return [v for v in range(self.n_nodes) if not ch[v]]

    def depth(self) -> List[int]:
        d = [0] * self.n_nodes
        for v in range(self.n_nodes):
            k, u = 0, v
            while self.parent[u] >= 0:
                u = self.parent[u]
                k += 1
            d[v] = k
        return d

    def path_tokens(self, v: int) -> int:
        t = 0
        while v >= 0:
            t += self.seg_len[v]
            v = self.parent[v]
        return t

    @property
    def n_expanded(self) -> int:
        return int(sum(self.path_tokens(l) for l in self.leaves()))

    def to_json(self) -> str:
        return json.dumps({"name": self.name, "parent": list(map(int, self.parent)),
                           "seg_len": list(map(int, self.seg_len))})

    @staticmethod
    def from_json(s: str) -> "Tree":
        d = json.loads(s)
        return Tree(d["name"], list(d["parent"]), list(d["seg_len"]))


# ---------------------------------------------------------------------------
# generators (seeded)
# ---------------------------------------------------------------------------

def tiny_binary_tree() -> Tree:
    """64-token prompt; two levels of binary branching with 32-token segments.

    Node ids: 0 root; 1, 2 its children; 3, 4 under 1; 5, 6 under 2.
    N = 64 + 2*32 + 4*32 = 256 compact tokens, 4 leaves.
    """
    return Tree("tiny_binary", [-1, 0, 0, 1, 1, 2, 2], [64, 32, 32, 32, 32, 32, 32])


def grpo_star_tree(seed: int = 2, prompt: int = 1024, group: int = 16,
                   lo: int = 256, hi: int = 1024) -> Tree:
    """One shared prompt with ``group`` sibling responses of U[lo, hi] tokens."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi + 1, size=group)
    return Tree("grpo_star", [-1] + [0] * group, [prompt] + [int(x) for x in lens])


def segment_tree(seed: int = 3, prompt: int = 512, seg: int = 256, levels: int = 4,
                 p_stop: float = 0.2, width: int = 16) -> Tree:
    """Binary segment tree with early stop and fallback.

    Level by level (1..levels) every live node spawns two children of ``seg``
    tokens.  Each non-root node stops (becomes a leaf) with probability
    ``p_stop``; a node at depth ``levels`` is a leaf.  Then, while the tree has
    fewer than ``width`` leaves, a uniformly chosen non-stopped node of depth
    < ``levels`` grows a fresh chain of ``seg``-token nodes down to depth
    ``levels``, which adds exactly one leaf.
    """
    rng = np.random.default_rng(seed)
    parent, seg_len, depth, stopped = [-1], [prompt], [0], [False]
    live = [0]
    for lvl in range(1, levels + 1):
        nxt = []
        for u in live:
            for _ in range(2):
                v = len(parent)
                parent.append(u)
                seg_len.append(seg)
                depth.append(lvl)
                st = bool(rng.random() < p_stop)
                stopped.append(st)
                if not st and lvl < levels:
                    nxt.append(v)
        live = nxt

    def n_leaves():
        has_child = [False] * len(parent)
        for v, p in enumerate(parent):
            if p >= 0:
                has_child[p] = True
        return sum(1 for h in has_child if not h)

    while n_leaves() < width:
        cand = [v for v in range(len(parent)) if not stopped[v] and depth[v] < levels]
        u = cand[int(rng.integers(0, len(cand)))]
        for lvl in range(depth[u] + 1, levels + 1):
            v = len(parent)
            parent.append(u)
            seg_len.append(seg)
            depth.append(lvl)
            stopped.append(False)
            u = v
    return Tree("segment_tree", parent, seg_len)


def agentic_tree(seed: int = 4, target: int = 65536, tol: float = 0.10,
                 ratio=(4.0, 6.0), median: int = 512, sigma: float = 1.0,
                 clip=(64, 4096), max_draws: int = 100000) -> Tree:
    """Irregular multi-turn tree, rejection-sampled.

    Each draw: depth D ~ U{2..8}; nodes are created breadth-first from the
    root; every node above depth D gets fan-out U{1..4}; a node at depth >= 2
    stops (no children) with probability 0.2.  Segment lengths are
    round(exp(N(ln median, sigma))) clipped to ``clip``.  A draw is accepted
    when the compact token count is within ``tol`` of ``target`` and the
    expanded/compact ratio lies in ``ratio``; otherwise the next draw comes
    from the same stream.
    """
    rng = np.random.default_rng(seed)
    lo_n, hi_n = target * (1 - tol), target * (1 + tol)

    def seglen():
        x = int(round(math.exp(rng.normal(math.log(median), sigma))))
        return min(max(x, clip[0]), clip[1])

    for _ in range(max_draws):
        D = int(rng.integers(2, 9))
        parent, seg_len, depth = [-1], [seglen()], [0]
        path = [seg_len[0]]
        frontier = [0]
        total = seg_len[0]
        too_big = False
        while frontier and not too_big:
            nxt = []
            for u in frontier:
                if depth[u] >= D:
                    continue
                if depth[u] >= 2 and rng.random() < 0.2:
                    continue
                fan = int(rng.integers(1, 5))
                for _c in range(fan):
                    v = len(parent)
                    L = seglen()
                    parent.append(u)
                    seg_len.append(L)
                    depth.append(depth[u] + 1)
                    path.append(path[u] + L)
                    total += L
                    nxt.append(v)
                    if total > hi_n:
                        too_big = True
                        break
                if too_big:
                    break
            frontier = nxt
        if too_big or total < lo_n:
            continue
        t = Tree("agentic_tree", parent, seg_len)
        r = t.n_expanded / t.n_tokens
        if ratio[0] <= r <= ratio[1]:
            return t
    raise RuntimeError("agentic_tree: no accepted draw")


def long_context_tree(seed: int = 5, prompt: int = 32768, branches: int = 64,
                      lo: int = 1024, hi: int = 8192) -> Tree:
    """A long shared prefix with ``branches`` chains of U{1..3} segments.

    Segment lengths are log-uniform in [lo, hi]: round(exp(U(ln lo, ln hi))).
    """
    rng = np.random.default_rng(seed)
    parent, seg_len = [-1], [prompt]
    for _ in range(branches):
        u = 0
        for _s in range(int(rng.integers(1, 4))):
            L = int(round(math.exp(rng.uniform(math.log(lo), math.log(hi)))))
            parent.append(u)
            seg_len.append(L)
            u = len(parent) - 1
    return Tree("long_context", parent, seg_len)


def chain_tree(lengths) -> Tree:
    """A single trajectory split into consecutive segments."""
    lengths = [int(x) for x in lengths]
    return Tree("chain", [-1] + list(range(len(lengths) - 1)), lengths)


def random_tree(rng: np.random.Generator, n_nodes: int, len_choices, n_roots: int = 1) -> Tree:
    """A random forest: node v > 0 picks a uniformly random earlier parent.

    The first ``n_roots`` nodes are roots.  Node ids are then shuffled so that
    children do not always have larger ids than their parents.
    """
    parent = [-1] * n_nodes
    for v in range(n_roots, n_nodes):
        parent[v] = int(rng.integers(0, v))
    lens = [int(rng.choice(len_choices)) for _ in range(n_nodes)]
    perm = rng.permutation(n_nodes)          # old id -> new id
    new_parent = [0] * n_nodes
    new_len = [0] * n_nodes
    for old in range(n_nodes):
        p = parent[old]
        new_parent[perm[old]] = -1 if p < 0 else int(perm[p])
        new_len[perm[old]] = lens[old]
    return Tree("random", new_parent, new_len)


def expanded_forest(t: Tree) -> Tree:
    """Each root-to-leaf trajectory as its own one-node tree (no sharing).

    Leaves in ascending id order; used to time the same kernels on the
    independent trajectories that dense training would process.
    """
    leaves = t.leaves()
    return Tree(t.name + "_expanded", [-1] * len(leaves), [t.path_tokens(l) for l in leaves])


# ---------------------------------------------------------------------------
# frozen fixtures
# ---------------------------------------------------------------------------

GENERATORS = {
    "tiny_binary": tiny_binary_tree,
    "grpo_star": grpo_star_tree,
    "segment_tree": segment_tree,
    "agentic_tree": agentic_tree,
    "long_context": long_context_tree,
}

# name -> (q heads, kv heads, head_dim); see tensors.py for the value recipes.
WORKLOADS = ["tiny_binary", "grpo_star", "segment_tree", "agentic_tree", "long_context"]


def load_tree(name: str) -> Tree:
    """Load a frozen tree fixture (written by ``make_trees.py``)."""
    path = os.path.join(TREE_DIR, name + ".json")
    with open(path) as f:
        return Tree.from_json(f.read())
