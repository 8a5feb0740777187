"""ctypes declarations of the C ABI in include/*.h (marshalling only)."""
from __future__ import annotations

import contextlib
import ctypes as C
import os

from . import build as _build

c_int32_p = C.POINTER(C.c_int32)
c_uint8_p = C.POINTER(C.c_uint8)
c_int64_p = C.POINTER(C.c_int64)


class PlanOpts(C.Structure):
    _fields_ = [("block", C.c_int32), ("bwd_chunk_qtiles", C.c_int32), ("bwd_cta_order", C.c_int32)]


class PlanInfo(C.Structure):
    _fields_ = [("n_tokens", C.c_int64), ("n_nodes", C.c_int32), ("block", C.c_int32),
                ("n_qtiles", C.c_int32), ("n_bwd_items", C.c_int32), ("n_pairs", C.c_int64),
                ("n_intervals", C.c_int64), ("n_tile_entries", C.c_int64), ("n_full_tiles", C.c_int64),
                ("n_split_kv_tiles", C.c_int32), ("bwd_chunk_qtiles", C.c_int32),
                ("n_partial_slots", C.c_int64)]


class PlanArrays(C.Structure):
    _fields_ = [("node_order", c_int32_p), ("node_off", c_int32_p), ("subend", c_int32_p),
                ("qi_ptr", c_int32_p), ("qi_lo", c_int32_p), ("qi_hi", c_int32_p),
                ("qt_ptr", c_int32_p), ("qt_kv", c_int32_p), ("qt_cls", c_uint8_p),
                ("kv_qlo", c_int32_p), ("kv_qhi", c_int32_p), ("fwd_order", c_int32_p),
                ("bwd_items", c_int32_p)]


# name -> (restype, argtypes); every symbol include/*.h declares
SIGNATURES = {
    "tree_attn_plan": (C.c_int, [c_int32_p, c_int32_p, C.c_int32, C.POINTER(PlanOpts), C.POINTER(C.c_void_p)]),
    "tree_attn_plan_info": (C.c_int, [C.c_void_p, C.POINTER(PlanInfo)]),
    "tree_attn_plan_export": (C.c_int, [C.c_void_p, C.POINTER(PlanArrays)]),
    "tree_attn_plan_upload": (C.c_int, [C.c_void_p]),
    "tree_attn_workspace_size": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_int32,
                                           C.POINTER(C.c_size_t), C.POINTER(C.c_size_t)]),
    "tree_attn_fwd": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                C.c_int32, C.c_int32, C.c_int32, C.c_float, C.c_void_p, C.c_size_t,
                                C.c_void_p]),
    "tree_attn_bwd": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32,
                                C.c_int32, C.c_float, C.c_void_p, C.c_size_t, C.c_void_p]),
    "tree_attn_bwd_stages": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                       C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32,
                                       C.c_int32, C.c_float, C.c_void_p, C.c_size_t, C.c_void_p, C.c_int32]),
    "tree_attn_bwd_noalloc": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                        C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32,
                                        C.c_int32, C.c_float, C.c_void_p]),
    "tree_attn_noalloc_scratch_bytes": (C.c_size_t, []),
    "tree_attn_get_device_status": (C.c_int, [C.c_void_p]),
    "tree_attn_selftest_wait_timeout": (C.c_int, [C.c_int32, C.c_void_p]),
    "tree_attn_debug_checks": (C.c_int, []),
    "tree_attn_selftest_bounds": (C.c_int, [C.c_void_p]),
    "tree_attn_plan_destroy": (None, [C.c_void_p]),
    "tree_attn_strerror": (C.c_char_p, [C.c_int]),
    # include/tree_batch.h
    "tree_attn_batch_work": (C.c_int, [C.c_int32, c_int32_p, c_int32_p, c_int32_p, c_int64_p, c_int64_p]),
    "tree_attn_batch_assign": (C.c_int, [C.c_int32, c_int64_p, C.c_int32, c_int32_p, c_int64_p]),
    "tree_attn_batch_microbatches": (C.c_int, [C.c_int32, c_int64_p, c_int64_p, c_int32_p, C.c_int32, C.c_int64,
                                               c_int32_p, c_int32_p]),
    "tree_attn_batch_forest": (C.c_int, [C.c_int32, c_int32_p, c_int32_p, c_int32_p, c_uint8_p, c_int32_p,
                                         c_int32_p, c_int32_p, c_int32_p]),
    # include/tree_linear.h
    "tree_attn_linear_workspace_size": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, c_int64_p,
                                                  C.POINTER(C.c_size_t)]),
    "tree_attn_linear_fwd": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                       C.c_int32, C.c_int32, C.c_int32, C.c_float, C.c_void_p, C.c_size_t,
                                       C.c_void_p]),
    "tree_attn_linear_bwd": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                       C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_int32,
                                       C.c_float, C.c_void_p, C.c_size_t, C.c_void_p]),
    # include/tree_loss.h
    "tree_attn_plan_trajectory_info": (C.c_int, [C.c_void_p, c_int32_p, c_int64_p]),
    "tree_attn_plan_trajectories": (C.c_int, [C.c_void_p, c_int32_p, c_int64_p, c_int32_p]),
    "tree_attn_plan_token_info": (C.c_int, [C.c_void_p, c_int32_p, c_int32_p]),
    "tree_attn_scale_rows": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int64, C.c_int64, C.c_void_p]),
    "tree_attn_traj_logprobs": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p,
                                          C.c_void_p]),
    "tree_attn_subtree_advantage": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_float, C.c_void_p,
                                              C.c_void_p, C.c_void_p, C.c_void_p]),
}

_LIB = None


def load(path: str = None) -> C.CDLL:
    """Load libtreeattn.so (built in-tree by ``build.build_library``).  Raises
    if it is missing: there is no fallback implementation."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    path = path or _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: run prefix_tree_attention_attn_gb300.build.build_library()")
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == _build.LIB:
        _LIB = lib
    return lib


@contextlib.contextmanager
def library(path: str):
    """Inside the block every call of the package goes to the library at
    ``path`` -- e.g. ``build.LIB_DEBUG``, the same kernels with their bounds
    checks compiled in.  Plans made inside the block belong to that library."""
    global _LIB
    saved = _LIB
    _LIB = load(path)
    try:
        yield _LIB
    finally:
        _LIB = saved


class TreeAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = load().tree_attn_strerror(status).decode()
        super().__init__(f"{what}: {msg} (status {status})")


def check(status: int, what: str) -> None:
    if status != 0:
        raise TreeAttnError(status, what)
