"""Linear attention over a packed rollout tree (``include/tree_linear.h``):
chunks of at most 128 tokens inside each node, the recurrent state carried
from every node into its children.  Marshalling only.

    o = tree_linear_fwd(plan, q, k, v, decay, scale)   # decay: fp32 [hkv] in (0, 1]
    dq, dk, dv = tree_linear_bwd(plan, q, k, v, do, decay, scale)
"""
from __future__ import annotations

import ctypes as C

from . import TreePlan, _check_tensor, _dptr, _stream_ptr
from . import _binding as B


def linear_workspace(plan: TreePlan, hkv: int, d: int):
    """(number of chunks, workspace bytes)."""
    nc, ws = C.c_int64(0), C.c_size_t(0)
    B.check(B.load().tree_attn_linear_workspace_size(plan.handle, hkv, d, C.byref(nc), C.byref(ws)),
            "tree_attn_linear_workspace_size")
    return int(nc.value), int(ws.value)


def tree_linear_fwd(plan: TreePlan, q, k, v, decay, scale: float, o=None, workspace=None, stream=None):
    """O [N, hq, d] bf16 = scale * sum over each token's path of gamma^(distance) (q.k) v."""
    import torch
    _, hq, d = q.shape
    hkv = k.shape[1]
    N = plan.n_tokens
    for name, t, shp in (("q", q, (N, hq, d)), ("k", k, (N, hkv, d)), ("v", v, (N, hkv, d))):
        _check_tensor(t, name, shp, torch.bfloat16)
    _check_tensor(decay, "decay", (hkv,), torch.float32)
    o = torch.empty_like(q) if o is None else o
    _check_tensor(o, "o", (N, hq, d), torch.bfloat16)
    _, need = linear_workspace(plan, hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    B.check(B.load().tree_attn_linear_fwd(plan.handle, _dptr(q), _dptr(k), _dptr(v), _dptr(o), _dptr(decay), hq, hkv,
                                          d, scale, _dptr(workspace), workspace.numel(), _stream_ptr(stream)),
            "tree_attn_linear_fwd")
    return o


def tree_linear_bwd(plan: TreePlan, q, k, v, do, decay, scale: float, dq=None, dk=None, dv=None, workspace=None,
                    stream=None):
    """dQ [N, hq, d], dK / dV [N, hkv, d] bf16 for the compact output gradient dO."""
    import torch
    _, hq, d = q.shape
    hkv = k.shape[1]
    N = plan.n_tokens
    for name, t, shp in (("q", q, (N, hq, d)), ("k", k, (N, hkv, d)), ("v", v, (N, hkv, d)),
                         ("do", do, (N, hq, d))):
        _check_tensor(t, name, shp, torch.bfloat16)
    _check_tensor(decay, "decay", (hkv,), torch.float32)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t, shp in (("dq", dq, (N, hq, d)), ("dk", dk, (N, hkv, d)), ("dv", dv, (N, hkv, d))):
        _check_tensor(t, name, shp, torch.bfloat16)
    _, need = linear_workspace(plan, hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    B.check(B.load().tree_attn_linear_bwd(plan.handle, _dptr(q), _dptr(k), _dptr(v), _dptr(do), _dptr(dq), _dptr(dk),
                                          _dptr(dv), _dptr(decay), hq, hkv, d, scale, _dptr(workspace),
                                          workspace.numel(), _stream_ptr(stream)),
            "tree_attn_linear_bwd")
    return dq, dk, dv
