"""Linear attention over a rollout tree, the slow and obvious way (test
infrastructure).

HARTS (abstract): hybrid models mix softmax attention with linear attention,
whose recurrent state must be carried from a shared prefix into every branch.
Our reading (the pages give no formula): per q-head h with kv-head
g = h // G and a per-kv-head decay gamma_g in (0, 1],

    o_i = scale * sum_{j on i's root-to-node path, j <= i} gamma^(pos_i - pos_j) (q_i . k_j) v_j

with pos the position along the trajectory (gamma = 1: plain causal linear
attention; gamma < 1: a retention-style decay).  Equivalently, the state
after token j of a trajectory, S_j = gamma S_(j-1) + k_j v_j^T, gives
o_i = scale * q_i^T S_i; at a branch point every child starts from its
parent's final state.

Two formulas, both fp64, on the expanded trajectories (one per leaf, first
copy of each compact token kept; the copies agree):
* ``forward_parallel`` -- the double sum above, as masked matrices;
* ``forward_recurrent`` -- the state recursion token by token.

``backward_recurrent`` is a second, independent formula on the compact tokens:
with S_t the state after token t (S_t = gamma S_prev(t) + k_t v_t^T, prev(t)
the token before t on its path), O_t = scale q_t^T S_t, and the adjoint
R_t = dL/dS_t = scale sum_h q_t^h dO_t^h^T + gamma sum_{u: prev(u) = t} R_u
(summed over every continuation of t: the next token of its node, or the first
token of each child node), so dQ_t = scale S_t dO_t, dK_t = R_t v_t and
dV_t = R_t^T k_t.

``backward_parallel`` gives the gradients of a scalar loss whose gradient with
respect to the compact O is dO, the same way the softmax oracle does: dO is
split over the copies of each token (any split that sums to dO gives the same
result, since every copy's output equals the compact one), and each
trajectory's part is differentiated in closed form.  With A = Q K^T and the
decay mask W, O = scale (A o W) V, so
    dV = scale (A o W)^T dO,  dA = scale (dO V^T) o W,  dQ = dA K,  dK = dA^T Q,
summed over the copies and, for dK and dV, over the q-heads of a kv-head.
"""
from __future__ import annotations

import numpy as np

from . import layout


def _as64(x):
    return np.asarray(x.float().numpy() if hasattr(x, "float") else x, dtype=np.float64)


def forward_parallel(parent, seg_len, q, k, v, decay, scale):
    """O [N, hq, d] (fp64).  q [N, hq, d], k / v [N, hkv, d], decay [hkv]."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    gam = np.asarray(decay, dtype=np.float64)
    N, hq, d = q.shape
    hkv = k.shape[1]
    G = hq // hkv
    out = np.full((N, hq, d), np.nan)
    for _, idx in layout.trajectories(parent, seg_len):
        L = len(idx)
        pos = np.arange(L)
        diff = pos[:, None] - pos[None, :]
        for h in range(hq):
            g = h // G
            w = np.where(diff >= 0, gam[g] ** np.maximum(diff, 0), 0.0)
            s = q[idx, h] @ k[idx, g].T
            o = scale * (s * w) @ v[idx, g]
            first = np.isnan(out[idx, h, 0])
            out[idx[first], h] = o[first]
    return out


def forward_recurrent(parent, seg_len, q, k, v, decay, scale):
    """The same output from the state recursion, one token at a time."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    gam = np.asarray(decay, dtype=np.float64)
    N, hq, d = q.shape
    hkv = k.shape[1]
    G = hq // hkv
    out = np.full((N, hq, d), np.nan)
    for _, idx in layout.trajectories(parent, seg_len):
        for g in range(hkv):
            S = np.zeros((d, d))
            for t in idx:
                S = gam[g] * S + np.outer(k[t, g], v[t, g])
                for h in range(g * G, (g + 1) * G):
                    if np.isnan(out[t, h, 0]):
                        out[t, h] = scale * (q[t, h] @ S)
    return out


def backward_parallel(parent, seg_len, q, k, v, do, decay, scale, split="multiplicity"):
    """dQ [N, hq, d], dK / dV [N, hkv, d] (fp64) for the compact gradient dO.

    ``split`` = "multiplicity": copy weight 1 / (trajectories holding the
    token); "first": all of a token's dO on its first trajectory (ascending
    leaf id).
    """
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    gam = np.asarray(decay, dtype=np.float64)
    N, hq, d = q.shape
    hkv = k.shape[1]
    G = hq // hkv
    if split == "multiplicity":
        w_tok = 1.0 / layout.multiplicity(parent, seg_len)
    elif split != "first":
        raise ValueError(split)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    seen = np.zeros(N, dtype=bool)
    for _, idx in layout.trajectories(parent, seg_len):
        L = len(idx)
        if split == "multiplicity":
            wt = w_tok[idx]
        else:
            wt = (~seen[idx]).astype(np.float64)
            seen[idx] = True
        diff = np.arange(L)[:, None] - np.arange(L)[None, :]
        for h in range(hq):
            g = h // G
            W = np.where(diff >= 0, gam[g] ** np.maximum(diff, 0), 0.0)
            Qt, Kt, Vt = q[idx, h], k[idx, g], v[idx, g]
            dOt = do[idx, h] * wt[:, None]
            M = (Qt @ Kt.T) * W
            dA = scale * (dOt @ Vt.T) * W
            np.add.at(dv[:, g], idx, scale * (M.T @ dOt))
            np.add.at(dq[:, h], idx, dA @ Kt)
            np.add.at(dk[:, g], idx, dA.T @ Qt)
    return dq, dk, dv


def backward_recurrent(parent, seg_len, q, k, v, do, decay, scale):
    """The same gradients from the state and adjoint recursions over the
    compact tokens (no trajectory expansion): states forward in packed order,
    adjoints backward, each token's adjoint summing over its continuations."""
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    gam = np.asarray(decay, dtype=np.float64)
    N, hq, d = q.shape
    hkv = k.shape[1]
    G = hq // hkv
    order, off, _ = layout.packed_layout(parent, seg_len)
    prev = np.full(N, -1, dtype=np.int64)       # token before t on its path
    for u in order:
        for m in range(seg_len[u]):
            t = off[u] + m
            if m > 0:
                prev[t] = t - 1
            elif parent[u] >= 0:
                prev[t] = off[parent[u]] + seg_len[parent[u]] - 1
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for g in range(hkv):
        S = np.zeros((N, d, d))
        for t in range(N):                      # parents come before children in packed order
            base = gam[g] * S[prev[t]] if prev[t] >= 0 else 0.0
            S[t] = base + np.outer(k[t, g], v[t, g])
        R = np.zeros((N, d, d))
        for t in range(N - 1, -1, -1):          # every continuation of t comes after t
            for h in range(g * G, (g + 1) * G):
                R[t] += scale * np.outer(q[t, h], do[t, h])
                dq[t, h] = scale * (S[t] @ do[t, h])
            if prev[t] >= 0:
                R[prev[t]] += gam[g] * R[t]
            dk[t, g] = R[t] @ v[t, g]
            dv[t, g] = R[t].T @ k[t, g]
    return dq, dk, dv
