"""GPU parity of the chunked tree linear attention (include/tree_linear.h)
against the fp64 oracle: relative Frobenius error <= 1e-2 per output (bf16
inputs and output, fp32 accumulation, the carried state rounded to bf16 as a
tensor-core operand)."""
import numpy as np
import pytest
import torch

from oracle import linear as OLN
from prefix_tree_attention_attn_gb300 import TreePlan, device_status
from prefix_tree_attention_attn_gb300.linear import linear_workspace, tree_linear_fwd
from workloads import tensors as WX
from workloads import trees as WT

pytestmark = pytest.mark.gpu

REL = 1e-2


@pytest.fixture(autouse=True)
def _lib(lib, cuda_device):
    yield
    torch.cuda.synchronize()
    assert device_status() == 0


def rel(got, want):
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30))


def check(t, hq, hkv, decay, seed):
    x = WX.draw_inputs(t.n_tokens, WX.HeadConfig(hq, hkv, 128), WX.ValueRecipe(1, 1, 1, 1, 1), seed)
    plan = TreePlan(t.parent, t.seg_len)
    dec = torch.tensor(decay, dtype=torch.float32)
    scale = 1 / np.sqrt(128)
    o = tree_linear_fwd(plan, x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), dec.cuda(), scale)
    torch.cuda.synchronize()
    want = OLN.forward_parallel(t.parent, t.seg_len, x["q"], x["k"], x["v"], decay, scale)
    got = o.float().cpu().numpy()
    for h in range(hq):
        e = rel(got[:, h], want[:, h])
        assert e <= REL, (h, e)
    return plan


@pytest.mark.parametrize("parent,seg_len,hq,hkv,decay", [
    ([-1], [1], 2, 1, [1.0]),
    ([-1], [300], 2, 2, [1.0, 0.98]),                          # several chunks in one node, ragged tail
    ([-1, 0, 0], [127, 129, 1], 4, 2, [0.95, 1.0]),            # chunk boundaries around 128
    ([-1, 0, 0, 1, 1, 2], [128, 200, 5, 64, 300, 33], 4, 1, [0.99]),
    ([-1, 0, 1, -1, 3], [70, 60, 5, 300, 2], 3, 3, [1.0, 0.9, 0.995]),   # forest, group 1
])
def test_small_trees(parent, seg_len, hq, hkv, decay):
    check(WT.Tree("s", parent, seg_len), hq, hkv, decay, 11)


@pytest.mark.parametrize("seed", range(3))
def test_random_trees(seed):
    rng = np.random.default_rng(300 + seed)
    t = WT.random_tree(rng, int(rng.integers(3, 12)), [1, 17, 127, 128, 129, 255], n_roots=1 + seed % 2)
    check(t, 4, 2, [0.97, 1.0], seed)


def test_segment_tree_workload():
    t = WT.load_tree("segment_tree")
    plan = check(t, 4, 1, [0.999], 5)
    nc, ws = linear_workspace(plan, 1, 128)
    assert nc == sum((L + 127) // 128 for L in t.seg_len)
