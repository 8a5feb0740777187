"""Loss-boundary calls (``include/tree_loss.h``): trajectory views of a plan,
per-token weights folded into a gradient, per-trajectory next-token log-probs
from compact logits, and subtree (segment-level) advantages.  Marshalling
only; the work runs in the library's kernels.

    mult, pos = token_info(plan)                       # host, [N] each
    dO_w = scale_rows(dO, w)                           # y[t] = x[t] * w[t]
    lse, lp = traj_logprobs(plan, logits, tokens)      # logits [N, V] bf16
    adv, node_c, tok_c = subtree_advantage(plan, rewards, flags=NORM_STD)
"""
from __future__ import annotations

import ctypes as C
from typing import Optional, Tuple

import numpy as np

from . import TreePlan, _check_tensor, _dptr, _stream_ptr
from . import _binding as B

NORM_STD = 1
SIZE_WEIGHTED = 2
NO_ROOT = 4


def trajectory_info(plan: TreePlan) -> Tuple[int, int]:
    """(number of trajectories = leaves, total trajectory tokens)."""
    nl, ne = C.c_int32(0), C.c_int64(0)
    B.check(B.load().tree_attn_plan_trajectory_info(plan.handle, C.byref(nl), C.byref(ne)),
            "tree_attn_plan_trajectory_info")
    return int(nl.value), int(ne.value)


def trajectories(plan: TreePlan) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """(leaf ids ascending, offsets [L+1], compact token of every trajectory position)."""
    nl, ne = trajectory_info(plan)
    leaves, ptr, tok = np.zeros(nl, np.int32), np.zeros(nl + 1, np.int64), np.zeros(max(ne, 1), np.int32)
    B.check(B.load().tree_attn_plan_trajectories(plan.handle, leaves.ctypes.data_as(B.c_int32_p),
                                                 ptr.ctypes.data_as(B.c_int64_p), tok.ctypes.data_as(B.c_int32_p)),
            "tree_attn_plan_trajectories")
    return leaves, ptr, tok[:ne]


def token_info(plan: TreePlan) -> Tuple[np.ndarray, np.ndarray]:
    """(multiplicity, position id) of every compact token, packed order."""
    N = plan.n_tokens
    mult, pos = np.zeros(N, np.int32), np.zeros(N, np.int32)
    B.check(B.load().tree_attn_plan_token_info(plan.handle, mult.ctypes.data_as(B.c_int32_p),
                                               pos.ctypes.data_as(B.c_int32_p)), "tree_attn_plan_token_info")
    return mult, pos


def scale_rows(x, w, out=None, stream=None):
    """out[t, ...] = x[t, ...] * w[t] (bf16 x / out, fp32 w; ``tree_attn_scale_rows``)."""
    import torch
    if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x: contiguous cuda bf16 expected")
    n = x.shape[0]
    _check_tensor(w, "w", (n,), torch.float32)
    out = torch.empty_like(x) if out is None else out
    _check_tensor(out, "out", tuple(x.shape), torch.bfloat16)
    row = x.numel() // max(n, 1)
    B.check(B.load().tree_attn_scale_rows(_dptr(x), _dptr(w), _dptr(out), n, row, _stream_ptr(stream)),
            "tree_attn_scale_rows")
    return out


def traj_logprobs(plan: TreePlan, logits, tokens, row_lse=None, out=None, stream=None):
    """(row logsumexp [N], next-token log-probs of every trajectory position
    [n_expanded - n_leaves]) from compact logits [N, V] bf16 and token ids [N] int32."""
    import torch
    N = plan.n_tokens
    V = logits.shape[1]
    _check_tensor(logits, "logits", (N, V), torch.bfloat16)
    _check_tensor(tokens, "tokens", (N,), torch.int32)
    nl, ne = trajectory_info(plan)
    row_lse = torch.empty(N, dtype=torch.float32, device=logits.device) if row_lse is None else row_lse
    out = torch.empty(ne - nl, dtype=torch.float32, device=logits.device) if out is None else out
    _check_tensor(row_lse, "row_lse", (N,), torch.float32)
    _check_tensor(out, "out", (ne - nl,), torch.float32)
    B.check(B.load().tree_attn_traj_logprobs(plan.handle, _dptr(logits), V, _dptr(tokens), _dptr(row_lse),
                                             _dptr(out) if out.numel() else None, _stream_ptr(stream)),
            "tree_attn_traj_logprobs")
    return row_lse, out


def subtree_advantage(plan: TreePlan, rewards, flags: int = 0, eps: float = 1e-6, stream=None):
    """(advantage of each trajectory, coefficient of each node by id, of each
    compact token) from per-trajectory rewards (leaves ascending id)."""
    import torch
    nl, _ = trajectory_info(plan)
    _check_tensor(rewards, "rewards", (nl,), torch.float32)
    dev = rewards.device
    adv = torch.empty(nl, dtype=torch.float32, device=dev)
    node_c = torch.empty(plan.info["n_nodes"], dtype=torch.float32, device=dev)
    tok_c = torch.empty(plan.n_tokens, dtype=torch.float32, device=dev)
    B.check(B.load().tree_attn_subtree_advantage(plan.handle, _dptr(rewards), flags, eps, _dptr(adv), _dptr(node_c),
                                                 _dptr(tok_c), _stream_ptr(stream)), "tree_attn_subtree_advantage")
    return adv, node_c, tok_c
