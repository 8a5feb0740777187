"""The forward and backward calls captured in a CUDA graph.

Once a plan's tables are on the device (its first call there, or
tree_attn_plan_upload), tree_attn_fwd and tree_attn_bwd allocate nothing and
do not synchronise, so a whole step can be captured once and replayed -- what
launch-bound small trees want (five launches per step become one).  Replays
must give the eager results: O, LSE, dK and dV bit for bit (dQ sums fp32
partials with atomics, so within 1e-3)."""
import numpy as np
import pytest
import torch

from prefix_tree_attention_attn_gb300 import TreePlan, device_status, tree_attn_bwd, tree_attn_fwd
from workloads import tensors as WX
from workloads import trees as WT

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny_binary", "grpo_star"])
def test_graph_replay_matches_eager(lib, cuda_device, name):
    t = WT.load_tree(name)
    heads, rec, xc = WX.workload_inputs(name, t.n_tokens)
    x = {k: v.to(cuda_device) for k, v in xc.items()}
    plan = TreePlan(t.parent, t.seg_len)
    plan.upload()
    o, lse = torch.empty_like(x["q"]), torch.empty((heads.hq, t.n_tokens), dtype=torch.float32, device=cuda_device)
    dq, dk, dv = torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"])
    ws = torch.empty(plan.workspace_size(heads.hq, heads.hkv, heads.d)[1], dtype=torch.uint8, device=cuda_device)

    def step():
        tree_attn_fwd(plan, x["q"], x["k"], x["v"], rec.scale, o=o, lse=lse)
        tree_attn_bwd(plan, x["q"], x["k"], x["v"], o, lse, x["do"], rec.scale, dq=dq, dk=dk, dv=dv, workspace=ws)

    step()
    torch.cuda.synchronize()
    eager = [a.clone() for a in (o, lse, dq, dk, dv)]
    for a in (o, lse, dq, dk, dv):
        a.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert device_status() == 0
    for nm, a, b in zip(("O", "LSE", "dQ", "dK", "dV"), (o, lse, dq, dk, dv), eager):
        assert torch.isfinite(a.float()).all(), nm
        if nm == "dQ":
            assert float((a.float() - b.float()).norm() / b.float().norm()) <= 1e-3
        else:
            assert torch.equal(a, b), nm
