"""The allocation-free backward (tree_attn_bwd_noalloc) against the regular one.

tree_attn_bwd_noalloc serves callers that cannot allocate device memory where
they run the backward -- their memory belongs to another allocator, or an
allocation could synchronise the device, or they work to a fixed budget.  It
keeps its scratch in one fixed device array of the library.  These tests call
it through the C ABI twice in a row on the same inputs (the second call must
not see anything left over from the first) and compare each result with the
regular entry point's, under the backward tolerance of the parity tests.  The
file sorts last so that a run stopping at the first failure has already run
every other test.
"""
import numpy as np
import pytest
import torch

from prefix_tree_attention_attn_gb300 import (TreePlan, device_status, noalloc_scratch_bytes, tree_attn_bwd,
                                              tree_attn_bwd_noalloc, tree_attn_fwd)
from prefix_tree_attention_attn_gb300 import _binding as B
from workloads import tensors as WX
from workloads import trees as WT

pytestmark = pytest.mark.gpu

BWD_REL = 1e-2     # relative Frobenius error per tensor, as in the parity tests


def rel(a, b):
    a = a.float()
    b = b.float()
    return float((a - b).norm() / b.norm().clamp_min(1e-30))


@pytest.mark.parametrize("parent,seg_len,hq,hkv,d", [
    ([-1, 0, 0, 1], [150, 90, 40, 33], 4, 2, 128),
    ([-1, 0, 0, 2], [200, 129, 64, 7], 2, 1, 64),
])
def test_noalloc_matches_regular_backward_twice(lib, cuda_device, parent, seg_len, hq, hkv, d):
    t = WT.Tree("noalloc", parent, seg_len)
    x = WX.draw_inputs(t.n_tokens, WX.HeadConfig(hq, hkv, d), WX.ValueRecipe(1, 1, 1, 1, 1), seed=77)
    scale = 1 / np.sqrt(d)
    plan = TreePlan(t.parent, t.seg_len)
    q, k, v, do = (x[n].to(cuda_device) for n in ("q", "k", "v", "do"))
    o, lse = tree_attn_fwd(plan, q, k, v, scale)
    ref = tree_attn_bwd(plan, q, k, v, o, lse, do, scale)
    torch.cuda.synchronize()
    for call in range(2):
        dq, dk, dv = (torch.full_like(a, float("nan")) for a in ref)
        tree_attn_bwd_noalloc(plan, q, k, v, o, lse, do, scale, dq, dk, dv)
        torch.cuda.synchronize()
        assert device_status() == 0
        for name, got, want in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
            assert torch.isfinite(got.float()).all(), (call, name)
            assert rel(got, want) <= BWD_REL, (call, name, rel(got, want))


def test_noalloc_rejects_problems_beyond_its_scratch(lib, cuda_device):
    # a single 70k-token segment with 4 q-heads needs > 32 MiB of fp32 dQ accumulator
    n_tok = 70000
    assert n_tok * 4 * 128 * 4 > noalloc_scratch_bytes()
    plan = TreePlan([-1], [n_tok])
    z = torch.zeros((n_tok, 4, 128), dtype=torch.bfloat16, device=cuda_device)
    zk = torch.zeros((n_tok, 2, 128), dtype=torch.bfloat16, device=cuda_device)
    lse = torch.zeros((4, n_tok), dtype=torch.float32, device=cuda_device)
    with pytest.raises(B.TreeAttnError) as err:
        tree_attn_bwd_noalloc(plan, z, zk, zk, z, lse, z, 1.0, torch.empty_like(z), torch.empty_like(zk),
                              torch.empty_like(zk))
    assert err.value.status == -11
