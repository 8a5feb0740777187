"""The bounds-checked build (libtreeattn_debug.so, -DTREE_ATTN_DEBUG) on the
GPU: every index the kernels take from the plan's tables or the tree's shape
(work items, kv-tile lists, subtree ends of partial and ragged tiles, partial
dK/dV slots, LSE / Delta rows, head numbers) is checked before it addresses
global memory; a failed check would set TREE_ATTN_ERR_DEVICE_BOUNDS - 1000 *
site in the status word and skip the access.  These tests run the adversarial
small trees (segment lengths 1, 127, 128, 129, 255; group sizes 1-4; d 64 and
128; forests) and larger trees through it, require a zero status and parity
with the fp64 oracle (or bit-identical results to the release build), and
check that a failing check is reported (self-test, no out-of-range access)."""
import numpy as np
import pytest
import torch

from prefix_tree_attention_attn_gb300 import TreePlan, build as _build, device_status, tree_attn_bwd, tree_attn_fwd
from prefix_tree_attention_attn_gb300 import _binding as B
from workloads import tensors as WX
from workloads import trees as WT

from .gpu_util import full_parity
from .test_gpu_parity import SMALL, draw

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def debug_lib(lib, cuda_device):
    path = _build.build_library(debug=True)
    dl = B.load(path)
    assert dl.tree_attn_debug_checks() == 1
    return path


def test_debug_selftest_reports_a_failed_check(debug_lib):
    with B.library(debug_lib) as dl:
        assert device_status() == 0
        assert dl.tree_attn_selftest_bounds(None) == 0
        st = device_status()
        assert st == -13 - 1000 * 98, st
        assert "bounds" in dl.tree_attn_strerror(st).decode()
        assert device_status() == 0          # read and cleared


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_debug_build_small_trees_clean_and_in_parity(debug_lib, case):
    parent, seg_len, hq, hkv, d = SMALL[case]
    t = WT.Tree("small", parent, seg_len)
    q, k, v, do = draw(t.n_tokens, hq, hkv, d, seed=case)
    with B.library(debug_lib):
        full_parity(t, q, k, v, do, 1 / np.sqrt(d), tag=f"debug case{case}")
        assert device_status() == 0


def run_both(t, heads, rec, x):
    out = []
    for path in (_build.LIB, _build.build_library(debug=True)):
        with B.library(path):
            plan = TreePlan(t.parent, t.seg_len)
            o, lse = tree_attn_fwd(plan, x["q"], x["k"], x["v"], rec.scale)
            dq, dk, dv = tree_attn_bwd(plan, x["q"], x["k"], x["v"], o, lse, x["do"], rec.scale)
            torch.cuda.synchronize()
            assert device_status() == 0, path
            out.append((o, lse, dq, dk, dv))
            plan.close()
    return out


@pytest.mark.parametrize("which", ["agentic_tree", "long_context_root_4_branches"])
def test_debug_build_large_trees_match_release_bitwise(debug_lib, which):
    """Large trees (the agentic tree; the long-context root with 4 branches at
    64 q-heads, whose backward takes the doubled chunk and the head-major CTA
    order): the checks pass and change no bit of O, LSE, dK, dV (dQ, summed
    with atomics, within 1e-3)."""
    if which == "agentic_tree":
        t = WT.load_tree(which)
        heads, rec = WX.HEADS[which], WX.VALUE_RECIPES[which]
    else:
        t = WT.long_context_tree(seed=WX.SEEDS["long_context"], branches=4)
        heads, rec = WX.HEADS["long_context"], WX.VALUE_RECIPES["long_context"]
    x = WX.draw_inputs(t.n_tokens, heads, rec, 1000 + WX.SEEDS.get(which, 5), device="cuda", chunk_rows=65536)
    (o1, l1, q1, k1, v1), (o2, l2, q2, k2, v2) = run_both(t, heads, rec, x)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    assert float((q1.float() - q2.float()).norm() / q1.float().norm()) <= 1e-3
