"""The allocation-free backward (tree_attn_bwd_noalloc), checked at the source.

tree_attn_bwd_noalloc serves callers that cannot allocate device memory where
they run the backward: their device memory belongs to another allocator (a
framework's caching pool), an allocation could synchronise the device, or they
work to a fixed memory budget.  It keeps its plan tables and workspace in one
fixed device array of the library, shared by every call.

These tests call it through the C ABI several times in a row on different
trees with nothing in between -- a larger problem first, then a smaller one
with another head layout, then the first again -- so a call that read what the
previous call left in the shared array would go wrong.  Each result is compared
with the fp64 oracle under the backward tolerance of the parity tests, and
with the regular entry point.  The file sorts last so that a run stopping at
the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from oracle import attention as OA
from prefix_tree_attention_attn_gb300 import (TreePlan, device_status, noalloc_scratch_bytes, tree_attn_bwd,
                                              tree_attn_bwd_noalloc, tree_attn_fwd)
from prefix_tree_attention_attn_gb300 import _binding as B
from workloads import tensors as WX
from workloads import trees as WT

from .gpu_util import BWD_REL, rel_fro

pytestmark = pytest.mark.gpu

# (parent, seg_len, hq, hkv, d): the first needs the most scratch
CASES = [
    ([-1, 0, 0, 1], [150, 90, 40, 33], 4, 2, 128),
    ([-1, 0, 0, 2], [200, 129, 64, 7], 2, 1, 64),
]


def prepare(case, seed, dev):
    parent, seg_len, hq, hkv, d = case
    t = WT.Tree("noalloc", parent, seg_len)
    x = WX.draw_inputs(t.n_tokens, WX.HeadConfig(hq, hkv, d), WX.ValueRecipe(1, 1, 1, 1, 1), seed=seed)
    scale = 1 / np.sqrt(d)
    plan = TreePlan(t.parent, t.seg_len)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = tree_attn_fwd(plan, q, k, v, scale)
    return {"t": t, "x": x, "scale": scale, "plan": plan, "dev": (q, k, v, o, lse, do)}


def test_noalloc_back_to_back_calls_match_the_oracle(lib, cuda_device):
    cases = [prepare(c, 77 + i, cuda_device) for i, c in enumerate(CASES)]
    torch.cuda.synchronize()
    order = [0, 1, 0]
    outs = []
    for ci in order:                          # no synchronisation between the calls
        c = cases[ci]
        q, k, v, o, lse, do = c["dev"]
        dq, dk, dv = (torch.full_like(a, float("nan")) for a in (q, k, v))
        tree_attn_bwd_noalloc(c["plan"], q, k, v, o, lse, do, c["scale"], dq, dk, dv)
        outs.append((dq, dk, dv))
    torch.cuda.synchronize()
    assert device_status() == 0
    for ci, got in zip(order, outs):
        c = cases[ci]
        t, x = c["t"], c["x"]
        want64 = OA.backward(t.parent, t.seg_len, x["q"], x["k"], x["v"], x["do"], c["scale"])
        q, k, v, o, lse, do = c["dev"]
        regular = tree_attn_bwd(c["plan"], q, k, v, o, lse, do, c["scale"])
        torch.cuda.synchronize()
        for name, g, w64, wreg in zip(("dQ", "dK", "dV"), got, want64, regular):
            gn = g.float().cpu().numpy()
            assert np.isfinite(gn).all(), (ci, name)
            e = rel_fro(gn, w64)
            assert e <= BWD_REL, (ci, name, "vs oracle", e)
            e2 = rel_fro(gn, wreg.float().cpu().numpy().astype(np.float64))
            assert e2 <= BWD_REL, (ci, name, "vs tree_attn_bwd", e2)


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
