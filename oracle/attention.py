"""fp64 reference attention over a rollout prefix tree (test infrastructure).

Definition followed (AReaL-DTA and HARTS abstracts: training on the shared
tree must give each root-to-leaf trajectory exactly what training it alone
gives):

* forward -- for every leaf, in ascending id order, gather the compact tokens
  of its root-to-leaf trajectory, and run dense causal softmax attention on
  that sequence:  S = scale * Q K^T, row r keeps keys c <= r, LSE = log sum
  exp(S), P = exp(S - LSE), O = P V.  A compact token takes the value from the
  first trajectory that contains it; every other copy must agree (a prefix
  token's causal output depends on its prefix only), which is checked.
* backward -- the compact dO is the gradient of one scalar loss; it is split
  over the copies of each token (weights summing to one: 1/multiplicity by
  default, or "all to the first trajectory"), each trajectory runs the
  textbook causal-attention VJP  dV = P^T dO,  dP = dO V^T,
  dS = P * (dP - rowsum(dO * O)),  dQ = scale dS K,  dK = scale dS^T Q,  and
  the results are scatter-added onto the compact tokens.
* grouped-query attention -- q-head h reads kv-head h // (Hq / Hkv); dK, dV
  sum over the q-heads of a group.

A second, independent formula (``masked_forward`` / ``masked_backward``)
works directly on the compact sequence with a dense mask built from ancestor
sets; it must agree with the expanded formula.

Layouts: Q, O, dO, dQ are [N, Hq, d]; K, V, dK, dV are [N, Hkv, d]; LSE is
[Hq, N] (natural log of the sum of exponentials of the scaled logits).  All
arithmetic is float64 on the CPU.
"""
from __future__ import annotations

from typing import Dict, Optional, Tuple

import numpy as np

from . import layout

_BLOCK_ELEMS = 1 << 23        # bound on one logits block (elements)


def _f64(x) -> np.ndarray:
    """Upcast a torch tensor (any dtype, CPU) or array to a float64 array."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def _rows_per_block(g: int, L: int) -> int:
    return int(max(16, min(L, _BLOCK_ELEMS // max(1, g * L))))


def causal_forward(q, k, v, scale: float) -> Tuple[np.ndarray, np.ndarray]:
    """Dense causal attention on one sequence.  q [L, Hq, d], k/v [L, Hkv, d].

    Returns O [L, Hq, d], LSE [Hq, L]."""
    L, hq, d = q.shape
    hkv = k.shape[1]
    g = hq // hkv
    O = np.zeros((L, hq, d))
    lse = np.zeros((hq, L))
    rb = _rows_per_block(g, L)
    for hk in range(hkv):
        Qg = q[:, hk * g:(hk + 1) * g, :].transpose(1, 0, 2)     # [g, L, d]
        Kh, Vh = k[:, hk, :], v[:, hk, :]
        for r0 in range(0, L, rb):
            r1 = min(L, r0 + rb)
            S = scale * (Qg[:, r0:r1, :] @ Kh[:r1].T)             # [g, rows, r1]
            rows = np.arange(r0, r1)[:, None]
            cols = np.arange(r1)[None, :]
            S = np.where(cols <= rows, S, -np.inf)
            m = S.max(axis=-1, keepdims=True)
            P = np.exp(S - m)
            l = P.sum(axis=-1, keepdims=True)
            lse[hk * g:(hk + 1) * g, r0:r1] = (m + np.log(l))[..., 0]
            O[r0:r1, hk * g:(hk + 1) * g, :] = ((P / l) @ Vh[:r1]).transpose(1, 0, 2)
    return O, lse


def causal_backward(q, k, v, o, lse, do, scale: float):
    """Textbook VJP of ``causal_forward``.  Returns dQ, dK, dV (fp64)."""
    L, hq, d = q.shape
    hkv = k.shape[1]
    g = hq // hkv
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    delta = (do * o).sum(axis=2).T                                   # rowsum(dO * O), [Hq, L]
    rb = _rows_per_block(g, L)
    for hk in range(hkv):
        hs = slice(hk * g, (hk + 1) * g)
        Qg = q[:, hs, :].transpose(1, 0, 2)
        dOg = do[:, hs, :].transpose(1, 0, 2)
        Kh, Vh = k[:, hk, :], v[:, hk, :]
        for r0 in range(0, L, rb):
            r1 = min(L, r0 + rb)
            S = scale * (Qg[:, r0:r1, :] @ Kh[:r1].T)
            rows = np.arange(r0, r1)[:, None]
            cols = np.arange(r1)[None, :]
            P = np.where(cols <= rows, np.exp(S - lse[hs, r0:r1, None]), 0.0)
            rows_g = g * (r1 - r0)
            # sum over the group's heads and the block's rows: P^T dO
            dv[:r1, hk, :] += P.transpose(2, 0, 1).reshape(r1, rows_g) @ dOg[:, r0:r1, :].reshape(rows_g, d)
            dP = dOg[:, r0:r1, :] @ Vh[:r1].T
            dS = P * (dP - delta[hs, r0:r1, None])
            dq[r0:r1, hs, :] = (scale * (dS @ Kh[:r1])).transpose(1, 0, 2)
            dk[:r1, hk, :] += scale * (dS.transpose(2, 0, 1).reshape(r1, rows_g) @ Qg[:, r0:r1, :].reshape(rows_g, d))
    return dq, dk, dv


def forward(parent, seg_len, q, k, v, scale: float, check_copies: bool = True,
            info: Optional[Dict] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Compact O [N, Hq, d] and LSE [Hq, N] by expanding every trajectory."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    N, hq, d = q.shape
    O = np.zeros_like(q)
    lse = np.zeros((hq, N))
    seen = np.zeros(N, dtype=bool)
    worst = 0.0
    for _, idx in layout.trajectories(parent, seg_len):
        o_t, l_t = causal_forward(q[idx], k[idx], v[idx], scale)
        old = seen[idx]
        if check_copies and old.any():
            worst = max(worst, float(np.abs(O[idx[old]] - o_t[old]).max()),
                        float(np.abs(lse[:, idx[old]] - l_t[:, old]).max()))
        new = idx[~old]
        O[new] = o_t[~old]
        lse[:, new] = l_t[:, ~old]
        seen[idx] = True
    if info is not None:
        info["copy_disagreement"] = worst
    if check_copies and worst > 1e-9:
        raise AssertionError(f"trajectory copies disagree by {worst}")
    return O, lse


def backward(parent, seg_len, q, k, v, do, scale: float, split: str = "multiplicity"):
    """Compact dQ, dK, dV by per-trajectory VJPs with dO split over copies.

    ``split`` = "multiplicity": copy weight 1/mult(t); "first": the whole
    dO of token t goes to the first trajectory (ascending leaf id) holding t.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    trajs = layout.trajectories(parent, seg_len)
    N = q.shape[0]
    if split == "multiplicity":
        w = 1.0 / layout.multiplicity(parent, seg_len)
    elif split != "first":
        raise ValueError(split)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    seen = np.zeros(N, dtype=bool)
    for _, idx in trajs:
        qt, kt, vt = q[idx], k[idx], v[idx]
        o_t, l_t = causal_forward(qt, kt, vt, scale)
        if split == "multiplicity":
            wt = w[idx]
        else:
            wt = (~seen[idx]).astype(np.float64)
            seen[idx] = True
        a, b, c = causal_backward(qt, kt, vt, o_t, l_t, do[idx] * wt[:, None, None], scale)
        np.add.at(dq, idx, a)
        np.add.at(dk, idx, b)
        np.add.at(dv, idx, c)
    return dq, dk, dv


# ---------------------------------------------------------------------------
# second formula: compact space, dense ancestor mask
# ---------------------------------------------------------------------------

def masked_forward(parent, seg_len, q, k, v, scale: float):
    """Masked softmax attention on the compact sequence (small N only)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    M = layout.dense_mask(parent, seg_len)
    N, hq, d = q.shape
    g = hq // k.shape[1]
    O = np.zeros_like(q)
    lse = np.zeros((hq, N))
    for h in range(hq):
        S = scale * (q[:, h, :] @ k[:, h // g, :].T)
        S = np.where(M, S, -np.inf)
        m = S.max(axis=1, keepdims=True)
        P = np.exp(S - m)
        l = P.sum(axis=1, keepdims=True)
        lse[h] = (m + np.log(l))[:, 0]
        O[:, h, :] = (P / l) @ v[:, h // g, :]
    return O, lse


def masked_backward(parent, seg_len, q, k, v, do, scale: float):
    """Textbook VJP of ``masked_forward`` with the full compact dO."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    M = layout.dense_mask(parent, seg_len)
    O, lse = masked_forward(parent, seg_len, q, k, v, scale)
    N, hq, d = q.shape
    g = hq // k.shape[1]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for h in range(hq):
        hk = h // g
        S = scale * (q[:, h, :] @ k[:, hk, :].T)
        P = np.where(M, np.exp(S - lse[h][:, None]), 0.0)
        dv[:, hk, :] += P.T @ do[:, h, :]
        dP = do[:, h, :] @ v[:, hk, :].T
        dS = P * (dP - (do[:, h, :] * O[:, h, :]).sum(axis=1, keepdims=True))
        dq[:, h, :] = scale * dS @ k[:, hk, :]
        dk[:, hk, :] += scale * dS.T @ q[:, h, :]
    return dq, dk, dv


# ---------------------------------------------------------------------------
# sampled evaluation for sizes where the full expansion is too expensive
# ---------------------------------------------------------------------------

def _row_keys(parent, seg_len, off, i: int, node: int) -> np.ndarray:
    """Compact key indices on token i's root-to-node path, causal in its own node."""
    parts = []
    for u in layout.root_path(parent, node):
        if u == node:
            parts.append(np.arange(off[u], i + 1))
        else:
            parts.append(np.arange(off[u], off[u] + seg_len[u]))
    return np.concatenate(parts)


def forward_rows(parent, seg_len, q, k, v, scale: float, rows, heads=None):
    """O and LSE of selected compact rows (each row's softmax over its own
    root-to-node path).  Returns O [len(rows), len(heads), d], LSE [len(heads), len(rows)]."""
    _, off, N = layout.packed_layout(parent, seg_len)
    tn = layout.token_nodes(parent, seg_len)
    hq = q.shape[1]
    g = hq // k.shape[1]
    heads = list(range(hq)) if heads is None else list(heads)
    O = np.zeros((len(rows), len(heads), q.shape[2]))
    lse = np.zeros((len(heads), len(rows)))
    for r, i in enumerate(rows):
        keys = _row_keys(parent, seg_len, off, int(i), int(tn[i]))
        qi = _f64(q[int(i)])
        kk = _f64(k[keys])
        vv = _f64(v[keys])
        for a, h in enumerate(heads):
            s = scale * (kk[:, h // g, :] @ qi[h])
            m = s.max()
            p = np.exp(s - m)
            l = p.sum()
            lse[a, r] = m + np.log(l)
            O[r, a] = (p / l) @ vv[:, h // g, :]
    return O, lse


def backward_rows_dq(parent, seg_len, q, k, v, do, scale: float, rows, heads=None):
    """dQ of selected compact rows: it depends on the row's own path only
    (dQ_i = scale * sum_j P_ij (dP_ij - dO_i . O_i) k_j), so it is exact here
    without expanding the tree."""
    _, off, N = layout.packed_layout(parent, seg_len)
    tn = layout.token_nodes(parent, seg_len)
    hq = q.shape[1]
    g = hq // k.shape[1]
    heads = list(range(hq)) if heads is None else list(heads)
    dQ = np.zeros((len(rows), len(heads), q.shape[2]))
    for r, i in enumerate(rows):
        keys = _row_keys(parent, seg_len, off, int(i), int(tn[i]))
        qi = _f64(q[int(i)])
        doi = _f64(do[int(i)])
        kk = _f64(k[keys])
        vv = _f64(v[keys])
        for a, h in enumerate(heads):
            s = scale * (kk[:, h // g, :] @ qi[h])
            p = np.exp(s - s.max())
            p /= p.sum()
            o = p @ vv[:, h // g, :]
            dp = vv[:, h // g, :] @ doi[h]
            ds = p * (dp - doi[h] @ o)
            dQ[r, a] = scale * (ds @ kk[:, h // g, :])
    return dQ


def backward_keys_dkdv(parent, seg_len, q, k, v, do, scale: float, keys, kv_heads=None):
    """dK, dV of selected compact keys.  Key j receives gradient from every
    query whose root-to-node path holds j (found by ancestor walking), so the
    cost per key is its number of descendants times their path lengths --
    cheap for keys near the end of a leaf segment.
    Returns dK, dV [len(keys), len(kv_heads), d]."""
    _, off, N = layout.packed_layout(parent, seg_len)
    tn = layout.token_nodes(parent, seg_len)
    A = layout.ancestor_matrix(parent)
    hq, hkv = q.shape[1], k.shape[1]
    g = hq // hkv
    kv_heads = list(range(hkv)) if kv_heads is None else list(kv_heads)
    d = q.shape[2]
    dK = np.zeros((len(keys), len(kv_heads), d))
    dV = np.zeros((len(keys), len(kv_heads), d))
    allrows = np.arange(N)
    for r, j in enumerate(keys):
        j = int(j)
        u = int(tn[j])
        desc = allrows[A[tn, u] & ((tn != u) | (allrows >= j))]
        kj = _f64(k[j])
        vj = _f64(v[j])
        for i in desc:
            keys_i = _row_keys(parent, seg_len, off, int(i), int(tn[i]))
            pos = int(np.searchsorted(keys_i, j))
            qi = _f64(q[int(i)])
            doi = _f64(do[int(i)])
            kk = _f64(k[keys_i])
            vv = _f64(v[keys_i])
            for a, hk in enumerate(kv_heads):
                for h in range(hk * g, (hk + 1) * g):
                    s = scale * (kk[:, hk, :] @ qi[h])
                    p = np.exp(s - s.max())
                    p /= p.sum()
                    o = p @ vv[:, hk, :]
                    dp_ij = doi[h] @ vj[hk]
                    ds_ij = p[pos] * (dp_ij - doi[h] @ o)
                    dV[r, a] += p[pos] * doi[h]
                    dK[r, a] += scale * ds_ij * qi[h]
    return dK, dV
