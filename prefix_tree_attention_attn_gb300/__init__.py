"""Prefix-tree attention for one GB300 (sm_103a): causal softmax attention,
forward and backward, over a packed rollout prefix tree.

Each shared prefix of the rollouts is stored once; every token attends exactly
to the tokens on its own root-to-node path, so each trajectory gets the
outputs and gradients it would get if trained on its own (AReaL-DTA and HARTS
abstracts).  The work runs in hand-written CUDA kernels behind a C ABI
(``include/tree_attn.h``, ``libtreeattn.so``); this module only marshals
arguments.  PyTorch supplies device memory and streams.

    plan = TreePlan(parent, seg_len)                 # host, C++ planner
    o, lse = tree_attn_fwd(plan, q, k, v, scale)     # q [N, hq, d] bf16 (cuda)
    dq, dk, dv = tree_attn_bwd(plan, q, k, v, o, lse, do, scale)

Tensors are token-major in packed order: node v's tokens are rows
``plan.node_off[v] : plan.node_off[v] + seg_len[v]``.
"""
from __future__ import annotations

import ctypes as C
from typing import Dict, Optional, Sequence

import numpy as np

from . import _binding as B

TILE_FULL = 1
TILE_PARTIAL = 2


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr_i32(a: np.ndarray):
    return a.ctypes.data_as(B.c_int32_p)


class TreePlan:
    """A plan for one rollout tree or forest (``tree_attn_plan``)."""

    def __init__(self, parent: Sequence[int], seg_len: Sequence[int], block: int = 0,
                 bwd_chunk_qtiles: int = 0, bwd_cta_order: int = 0):
        self._lib = B.load()
        self._h = None
        par, sl = _i32(parent), _i32(seg_len)
        if par.ndim != 1 or sl.shape != par.shape:
            raise ValueError("parent and seg_len must be 1-D arrays of equal length")
        opts = B.PlanOpts(block, bwd_chunk_qtiles, bwd_cta_order)
        h = C.c_void_p()
        B.check(self._lib.tree_attn_plan(_ptr_i32(par), _ptr_i32(sl), len(par), C.byref(opts), C.byref(h)),
                "tree_attn_plan")
        self._h = h
        self.seg_len = sl
        inf = B.PlanInfo()
        B.check(self._lib.tree_attn_plan_info(h, C.byref(inf)), "tree_attn_plan_info")
        self.info = {f: getattr(inf, f) for f, _ in B.PlanInfo._fields_}
        self.n_tokens = int(inf.n_tokens)
        self.n_pairs = int(inf.n_pairs)
        self.node_off = self.export(("node_off",))["node_off"]

    @property
    def handle(self):
        return self._h

    def export(self, fields: Optional[Sequence[str]] = None) -> Dict[str, np.ndarray]:
        """Copies of the plan arrays (``tree_attn_plan_export``)."""
        i = self.info
        sizes = {"node_order": i["n_nodes"], "node_off": i["n_nodes"], "subend": i["n_tokens"],
                 "qi_ptr": i["n_qtiles"] + 1, "qi_lo": i["n_intervals"], "qi_hi": i["n_intervals"],
                 "qt_ptr": i["n_qtiles"] + 1, "qt_kv": i["n_tile_entries"], "qt_cls": i["n_tile_entries"],
                 "kv_qlo": i["n_qtiles"], "kv_qhi": i["n_qtiles"], "fwd_order": i["n_qtiles"],
                 "bwd_items": 4 * i["n_bwd_items"]}
        fields = list(sizes) if fields is None else list(fields)
        out, arr = {}, B.PlanArrays()
        for f in fields:
            dt = np.uint8 if f == "qt_cls" else np.int32
            a = np.zeros(max(1, int(sizes[f])), dtype=dt)
            out[f] = a
            setattr(arr, f, a.ctypes.data_as(B.c_uint8_p if f == "qt_cls" else B.c_int32_p))
        B.check(self._lib.tree_attn_plan_export(self._h, C.byref(arr)), "tree_attn_plan_export")
        return {f: out[f][:int(sizes[f])] for f in fields}

    def upload(self) -> None:
        B.check(self._lib.tree_attn_plan_upload(self._h), "tree_attn_plan_upload")

    def workspace_size(self, hq: int, hkv: int, d: int):
        f, b = C.c_size_t(), C.c_size_t()
        B.check(self._lib.tree_attn_workspace_size(self._h, hq, hkv, d, C.byref(f), C.byref(b)),
                "tree_attn_workspace_size")
        return int(f.value), int(b.value)

    def close(self) -> None:
        if self._h is not None:
            self._lib.tree_attn_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _stream_ptr(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def _dptr(t) -> C.c_void_p:
    return C.c_void_p(t.data_ptr())


def _check_tensor(t, name, shape, dtype):
    import torch
    if not t.is_cuda or t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError(f"{name}: expected contiguous cuda {dtype} {tuple(shape)}, got "
                         f"{t.device} {t.dtype} {tuple(t.shape)}")


def tree_attn_fwd(plan: TreePlan, q, k, v, softmax_scale: float, o=None, lse=None, stream=None):
    """O [N, hq, d] bf16 and LSE [hq, N] fp32 (``tree_attn_fwd``)."""
    import torch
    N, hq, d = q.shape
    hkv = k.shape[1]
    _check_tensor(q, "q", (plan.n_tokens, hq, d), torch.bfloat16)
    _check_tensor(k, "k", (plan.n_tokens, hkv, d), torch.bfloat16)
    _check_tensor(v, "v", (plan.n_tokens, hkv, d), torch.bfloat16)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((hq, N), dtype=torch.float32, device=q.device)
    _check_tensor(o, "o", q.shape, torch.bfloat16)
    _check_tensor(lse, "lse", (hq, N), torch.float32)
    B.check(B.load().tree_attn_fwd(plan.handle, _dptr(q), _dptr(k), _dptr(v), _dptr(o), _dptr(lse), hq, hkv, d,
                                   float(softmax_scale), None, 0, _stream_ptr(stream)), "tree_attn_fwd")
    return o, lse


BWD_PRE, BWD_MAIN, BWD_POST = 1, 2, 4


def tree_attn_bwd(plan: TreePlan, q, k, v, o, lse, dout, softmax_scale: float, dq=None, dk=None, dv=None,
                  workspace=None, stream=None, stages: int = 7):
    """dQ, dK, dV (bf16) from the forward's O and LSE and the output gradient.
    ``stages`` (bit mask of BWD_PRE / BWD_MAIN / BWD_POST) runs part of the
    backward (``tree_attn_bwd_stages``); stages must run in order with one
    workspace."""
    import torch
    _, hq, d = q.shape
    hkv = k.shape[1]
    N = plan.n_tokens
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_bwd_tensors(N, hq, hkv, d, q=q, k=k, v=v, o=o, lse=lse, dout=dout, dq=dq, dk=dk, dv=dv)
    _, need = plan.workspace_size(hq, hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    args = (plan.handle, _dptr(q), _dptr(k), _dptr(v), _dptr(o), _dptr(lse), _dptr(dout), _dptr(dq), _dptr(dk),
            _dptr(dv), hq, hkv, d, float(softmax_scale), _dptr(workspace), workspace.numel(), _stream_ptr(stream))
    if int(stages) == BWD_PRE | BWD_MAIN | BWD_POST:
        B.check(B.load().tree_attn_bwd(*args), "tree_attn_bwd")
    else:
        B.check(B.load().tree_attn_bwd_stages(*args, int(stages)), "tree_attn_bwd_stages")
    return dq, dk, dv


def _check_bwd_tensors(N, hq, hkv, d, **t):
    """Every backward tensor against the plan's token count N and the head
    layout, before anything is launched (the library sizes its reads and
    writes from the plan)."""
    import torch
    shapes = {"q": (N, hq, d), "k": (N, hkv, d), "v": (N, hkv, d), "o": (N, hq, d), "lse": (hq, N),
              "dout": (N, hq, d), "dq": (N, hq, d), "dk": (N, hkv, d), "dv": (N, hkv, d)}
    for name, x in t.items():
        _check_tensor(x, name, shapes[name], torch.float32 if name == "lse" else torch.bfloat16)


def tree_attn_bwd_noalloc(plan: TreePlan, q, k, v, o, lse, dout, softmax_scale: float, dq, dk, dv, stream=None):
    """Backward into caller-provided dq / dk / dv without allocating anything
    (``tree_attn_bwd_noalloc``): for callers that cannot allocate device memory
    at this point, because another allocator owns it, because allocation could
    synchronise the device, or because of a fixed memory budget.  The library's
    fixed scratch (``noalloc_scratch_bytes()``) bounds the problem size, and
    calls that overlap on the GPU share that scratch, so run them one after
    another."""
    _, hq, d = q.shape
    hkv = k.shape[1]
    _check_bwd_tensors(plan.n_tokens, hq, hkv, d, q=q, k=k, v=v, o=o, lse=lse, dout=dout, dq=dq, dk=dk, dv=dv)
    B.check(B.load().tree_attn_bwd_noalloc(plan.handle, _dptr(q), _dptr(k), _dptr(v), _dptr(o), _dptr(lse),
                                           _dptr(dout), _dptr(dq), _dptr(dk), _dptr(dv), hq, hkv, d,
                                           float(softmax_scale), _stream_ptr(stream)), "tree_attn_bwd_noalloc")
    return dq, dk, dv


def noalloc_scratch_bytes() -> int:
    """Bytes of the fixed device scratch that ``tree_attn_bwd_noalloc`` uses."""
    return int(B.load().tree_attn_noalloc_scratch_bytes())


def device_status(stream=None) -> int:
    """Synchronise and read/clear the kernels' device status word (0 = fine)."""
    return int(B.load().tree_attn_get_device_status(_stream_ptr(stream)))
