"""The C-ABI library loads, exports every symbol include/*.h declares, and
rejects bad arguments on the host (CPU only; no compute call is made)."""
import ctypes as C
import os
import re

import numpy as np
import pytest

from prefix_tree_attention_attn_gb300 import _binding as B
from prefix_tree_attention_attn_gb300 import TreePlan

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
HEADER = os.path.join(INCLUDE, "tree_attn.h")


def declared_functions():
    text = "".join(open(os.path.join(INCLUDE, f)).read() for f in sorted(os.listdir(INCLUDE)) if f.endswith(".h"))
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tree_attn_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
        assert n in B.SIGNATURES, n


def test_status_codes_named(lib):
    text = open(HEADER).read()
    codes = {int(v) for v in re.findall(r"#define TREE_ATTN_(?:OK|ERR_[A-Z_]+)\s+(-?\d+)", text)}
    assert codes == set(range(-13, 1))
    for code in codes:
        s = lib.tree_attn_strerror(code).decode()
        assert s and s != "unknown status"
    assert lib.tree_attn_strerror(-10 - 1000 * 5).decode().startswith("a bounded device wait")


def plan_status(lib, parent, seg_len, block=0, chunk=0):
    par = np.asarray(parent, dtype=np.int32)
    sl = np.asarray(seg_len, dtype=np.int32)
    h = C.c_void_p()
    opts = B.PlanOpts(block, chunk, 0)
    st = lib.tree_attn_plan(par.ctypes.data_as(B.c_int32_p), sl.ctypes.data_as(B.c_int32_p), len(par),
                            C.byref(opts), C.byref(h))
    if st == 0:
        lib.tree_attn_plan_destroy(h)
    return st


@pytest.mark.parametrize("parent,seg_len,code", [
    ([-1, 0], [3, 0], -2),            # empty segment
    ([-1, 0], [3, -1], -2),
    ([0], [3], -2),                   # self parent
    ([-1, 5], [3, 3], -2),            # parent out of range
    ([-1, -2], [3, 3], -2),
    ([1, 0], [2, 2], -2),             # cycle, no root
    ([-1, 2, 1], [1, 2, 2], -2),      # cycle beside a root
    ([], [], -1),
])
def test_invalid_trees_rejected(lib, parent, seg_len, code):
    assert plan_status(lib, parent, seg_len) == code


def test_invalid_options_and_sizes(lib):
    assert plan_status(lib, [-1], [4], block=-3) == -1
    assert plan_status(lib, [-1], [4], block=2048) == -1
    assert plan_status(lib, [-1], [4], chunk=-1) == -1
    for bad in (-1, 3):
        par, sl, h = np.asarray([-1], dtype=np.int32), np.asarray([4], dtype=np.int32), C.c_void_p()
        assert lib.tree_attn_plan(par.ctypes.data_as(B.c_int32_p), sl.ctypes.data_as(B.c_int32_p), 1,
                                  C.byref(B.PlanOpts(0, 0, bad)), C.byref(h)) == -1
    assert plan_status(lib, [-1, 0], [2**30, 2**30]) == -3      # token count overflows int32
    h = C.c_void_p()
    assert lib.tree_attn_plan(None, None, 1, None, C.byref(h)) == -1
    assert lib.tree_attn_plan_info(None, None) == -1
    assert lib.tree_attn_plan_export(None, None) == -1


def test_compute_calls_validate_before_touching_the_device(lib):
    p = TreePlan([-1, 0], [100, 60])
    # null tensors -> invalid argument, checked on the host first
    assert lib.tree_attn_fwd(p.handle, None, None, None, None, None, 2, 2, 64, 1.0, None, 0, None) == -1
    assert lib.tree_attn_bwd(p.handle, None, None, None, None, None, None, None, None, None,
                             2, 2, 64, 1.0, None, 0, None) == -1
    # unsupported head configurations
    f, b = C.c_size_t(), C.c_size_t()
    assert lib.tree_attn_workspace_size(p.handle, 3, 2, 64, C.byref(f), C.byref(b)) == -4
    assert lib.tree_attn_workspace_size(p.handle, 4, 2, 96, C.byref(f), C.byref(b)) == -4
    assert lib.tree_attn_workspace_size(p.handle, 4, 2, 128, C.byref(f), C.byref(b)) == 0
    assert f.value == 0 and b.value > 0
    p64 = TreePlan([-1, 0], [100, 60], block=64)
    assert lib.tree_attn_workspace_size(p64.handle, 4, 2, 128, C.byref(f), C.byref(b)) == -4
    # misaligned device pointers are refused before any launch
    fake = C.c_void_p(0x1000)
    odd = C.c_void_p(0x1008)
    assert lib.tree_attn_fwd(p.handle, odd, fake, fake, fake, fake, 2, 2, 64, 1.0, None, 0, None) == -5
    assert lib.tree_attn_fwd(p.handle, fake, fake, fake, fake, fake, 2, 2, 64, float("nan"),
                             None, 0, None) == -1
    assert lib.tree_attn_fwd(p.handle, fake, fake, fake, fake, fake, 2, 2, 64, -0.5, None, 0, None) == -1
    assert lib.tree_attn_bwd(p.handle, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                             2, 2, 64, 0.0, fake, 1 << 30, None) == -1
    # workspace too small
    assert lib.tree_attn_bwd(p.handle, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                             2, 2, 64, 1.0, fake, 16, None) == -6


def test_linear_calls_validate_on_the_host(lib):
    """The linear-attention calls refuse bad arguments before any device work."""
    p = TreePlan([-1, 0], [100, 60])
    fake, odd = C.c_void_p(0x1000), C.c_void_p(0x1008)
    f7 = [fake] * 7
    bwd = lib.tree_attn_linear_bwd
    fwd = lib.tree_attn_linear_fwd
    assert bwd(p.handle, None, *f7[:6], fake, 2, 1, 128, 1.0, fake, 1 << 30, None) == -1      # null tensor
    assert bwd(p.handle, *f7, None, 2, 1, 128, 1.0, fake, 1 << 30, None) == -1                # null decay
    assert bwd(p.handle, *f7, fake, 3, 2, 128, 1.0, fake, 1 << 30, None) == -1                # hq % hkv != 0
    assert bwd(p.handle, *f7, fake, 2, 1, 64, 1.0, fake, 1 << 30, None) == -4                 # d != 128
    assert bwd(p.handle, *f7, fake, 2, 1, 128, 0.0, fake, 1 << 30, None) == -1                # scale <= 0
    assert bwd(p.handle, *f7, fake, 2, 1, 128, float("inf"), fake, 1 << 30, None) == -1
    assert bwd(p.handle, odd, *f7[:6], fake, 2, 1, 128, 1.0, fake, 1 << 30, None) == -5      # misaligned q
    assert bwd(p.handle, *f7[:6], odd, fake, 2, 1, 128, 1.0, fake, 1 << 30, None) == -5      # misaligned dv
    assert fwd(p.handle, None, fake, fake, fake, fake, 2, 1, 128, 1.0, fake, 1 << 30, None) == -1
    assert fwd(p.handle, fake, fake, fake, fake, fake, 2, 1, 64, 1.0, fake, 1 << 30, None) == -4
    assert fwd(p.handle, fake, fake, odd, fake, fake, 2, 1, 128, 1.0, fake, 1 << 30, None) == -5


class FakeCudaTensor:
    """Stands in for a device tensor so that the binding's host-side checks
    run on a machine without a GPU; nothing is ever launched with it."""

    def __init__(self, shape, dtype):
        self.shape, self.dtype, self.is_cuda, self.device = tuple(shape), dtype, True, "cuda:0"

    def is_contiguous(self):
        return True

    def data_ptr(self):
        raise AssertionError("the binding reached a launch with a mismatched tensor")


def test_tensors_must_match_the_plan_before_any_launch(lib):
    """Every compute wrapper checks each tensor against the plan's token count
    (the library sizes its reads and writes from the plan): a q shorter or
    longer than the plan is refused with ValueError, before any launch."""
    import torch
    from prefix_tree_attention_attn_gb300 import tree_attn_bwd, tree_attn_bwd_noalloc, tree_attn_fwd
    from prefix_tree_attention_attn_gb300.linear import tree_linear_bwd, tree_linear_fwd
    p = TreePlan([-1, 0], [100, 60])          # 160 tokens
    hq, hkv, d = 4, 2, 128
    bf, f32 = torch.bfloat16, torch.float32
    for n_q in (159, 161, 320):
        def t(n, h):
            return FakeCudaTensor((n, h, d), bf)
        good_q, bad_q = t(160, hq), t(n_q, hq)
        kk, vv = t(160, hkv), t(160, hkv)
        lse = FakeCudaTensor((hq, 160), f32)
        outs = dict(dq=t(160, hq), dk=t(160, hkv), dv=t(160, hkv))
        with pytest.raises(ValueError):
            tree_attn_fwd(p, bad_q, kk, vv, 1.0, o=t(n_q, hq), lse=FakeCudaTensor((hq, n_q), f32))
        with pytest.raises(ValueError):
            tree_attn_bwd(p, bad_q, kk, vv, t(n_q, hq), lse, t(n_q, hq), 1.0, workspace=good_q, **outs)
        with pytest.raises(ValueError):      # right q, short dout
            tree_attn_bwd(p, good_q, kk, vv, good_q, lse, t(n_q, hq), 1.0, workspace=good_q, **outs)
        with pytest.raises(ValueError):      # right inputs, dq of another length
            tree_attn_bwd(p, good_q, kk, vv, good_q, lse, good_q, 1.0, dq=t(n_q, hq), dk=outs["dk"],
                          dv=outs["dv"], workspace=good_q)
        with pytest.raises(ValueError):
            tree_attn_bwd_noalloc(p, bad_q, kk, vv, t(n_q, hq), lse, t(n_q, hq), 1.0, **outs)
        dec = FakeCudaTensor((hkv,), f32)
        with pytest.raises(ValueError):
            tree_linear_fwd(p, bad_q, kk, vv, dec, 1.0, o=t(n_q, hq), workspace=good_q)
        with pytest.raises(ValueError):
            tree_linear_bwd(p, bad_q, kk, vv, t(n_q, hq), dec, 1.0, workspace=good_q, **outs)


def test_debug_build_flags(lib):
    """The release library carries no bounds checks (its self-test refuses);
    the twin built with -DTREE_ATTN_DEBUG says it has them."""
    from prefix_tree_attention_attn_gb300 import build as _build
    assert lib.tree_attn_debug_checks() == 0
    assert lib.tree_attn_selftest_bounds(None) == -4
    dl = B.load(_build.build_library(debug=True))
    assert dl.tree_attn_debug_checks() == 1
    assert lib.tree_attn_strerror(-13 - 1000 * 211).decode() == "a debug bounds check failed"
    assert lib.tree_attn_strerror(-10 - 1000 * 67).decode() == "a bounded device wait ran out"
