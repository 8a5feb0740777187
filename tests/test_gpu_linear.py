"""GPU parity of the chunked tree linear attention (include/tree_linear.h)
against the fp64 oracle: relative Frobenius error <= 1e-2 per output (bf16
inputs and output, fp32 accumulation, the carried state rounded to bf16 as a
tensor-core operand)."""
import numpy as np
import pytest
import torch

from oracle import linear as OLN
from prefix_tree_attention_attn_gb300 import TreePlan, device_status
from prefix_tree_attention_attn_gb300.linear import linear_workspace, tree_linear_bwd, tree_linear_fwd
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
    # a star: the children's first chunks fall in later batches of the scan than
    # the root's last one
    ([-1] + [0] * 20, [300] + [(17 * i) % 260 + 1 for i in range(20)], 4, 2, [0.99, 1.0]),
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


# --------------------------------------------------------------------------
# backward: dQ (the forward with (dO, V, K)), dK and dV (the reverse adjoint
# scan) against the fp64 oracle's per-trajectory VJP
# --------------------------------------------------------------------------

def check_bwd(t, hq, hkv, decay, seed):
    x = WX.draw_inputs(t.n_tokens, WX.HeadConfig(hq, hkv, 128), WX.ValueRecipe(1, 1, 1, 1, 1), seed)
    plan = TreePlan(t.parent, t.seg_len)
    dec = torch.tensor(decay, dtype=torch.float32)
    scale = 1 / np.sqrt(128)
    dq, dk, dv = tree_linear_bwd(plan, x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["do"].cuda(), dec.cuda(),
                                 scale)
    torch.cuda.synchronize()
    want = OLN.backward_parallel(t.parent, t.seg_len, x["q"], x["k"], x["v"], x["do"], decay, scale)
    for name, g, w in zip(("dq", "dk", "dv"), (dq, dk, dv), want):
        got = g.float().cpu().numpy()
        for h in range(got.shape[1]):
            e = rel(got[:, h], w[:, h])
            assert e <= REL, (name, h, e)


@pytest.mark.parametrize("parent,seg_len,hq,hkv,decay", [
    ([-1], [1], 2, 1, [1.0]),
    ([-1], [300], 2, 2, [1.0, 0.98]),
    ([-1, 0, 0], [127, 129, 1], 4, 2, [0.95, 1.0]),
    ([-1, 0, 0, 1, 1, 2], [128, 200, 5, 64, 300, 33], 4, 1, [0.99]),
    ([-1, 0, 1, -1, 3], [70, 60, 5, 300, 2], 3, 3, [1.0, 0.9, 0.995]),
    ([-1] + [0] * 20, [300] + [(17 * i) % 260 + 1 for i in range(20)], 4, 2, [0.99, 1.0]),   # star
])
def test_bwd_small_trees(parent, seg_len, hq, hkv, decay):
    check_bwd(WT.Tree("s", parent, seg_len), hq, hkv, decay, 21)


@pytest.mark.parametrize("seed", range(2))
def test_bwd_random_trees(seed):
    rng = np.random.default_rng(400 + seed)
    t = WT.random_tree(rng, int(rng.integers(3, 10)), [1, 17, 127, 128, 129, 255], n_roots=1 + seed % 2)
    check_bwd(t, 4, 2, [0.97, 1.0], 40 + seed)


def test_deep_chain_uses_the_one_walk_scans():
    # 40 nested nodes: deeper than the depth-by-depth scans take, so both scans
    # walk every chunk in one pass
    t = WT.Tree("deep", [-1] + list(range(39)), [(37 * i) % 150 + 1 for i in range(40)])
    check(t, 4, 2, [0.99, 0.97], 81)
    check_bwd(t, 4, 2, [0.99, 0.97], 82)


def test_persistent_kernels_walk_several_chunks():
    # 16 kv-heads leave 9 chunk lanes on a 152-SM GPU, so each CTA of the output
    # and dK/dV kernels walks several chunks of ragged lengths (the next chunk's
    # K, V and state load while the current one runs)
    t = WT.Tree("wide", [-1] + [0] * 6, [640, 700, 333, 129, 517, 256, 901])
    nc, _ = linear_workspace(TreePlan(t.parent, t.seg_len), 16, 128)
    assert nc >= 3 * (torch.cuda.get_device_properties(0).multi_processor_count // 16)
    decay = [0.97 + 0.002 * i for i in range(16)]
    check(t, 32, 16, decay, 91)
    check_bwd(t, 32, 16, decay, 92)


@pytest.mark.parametrize("seed", range(2))
def test_many_nodes(seed):
    # 40 to 60 short nodes: node boundaries at every position of the scans' batches
    rng = np.random.default_rng(500 + seed)
    t = WT.random_tree(rng, int(rng.integers(40, 61)), [1, 17, 129], n_roots=1 + seed)
    check(t, 2, 1, [0.98], 60 + seed)
    check_bwd(t, 2, 1, [0.98], 70 + seed)


def test_bwd_timing_segment_tree():
    """Times one backward on the segment tree (32 q-heads, 8 kv-heads) and
    checks the outputs are finite; the parity cases above pin the values."""
    t = WT.load_tree("segment_tree")
    x = WX.draw_inputs(t.n_tokens, WX.HeadConfig(32, 8, 128), WX.ValueRecipe(1, 1, 1, 1, 1), 9, device="cuda")
    plan = TreePlan(t.parent, t.seg_len)
    dec = torch.full((8,), 0.999, dtype=torch.float32, device="cuda")
    _, need = linear_workspace(plan, 8, 128)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    args = (plan, x["q"], x["k"], x["v"], x["do"], dec, 1 / np.sqrt(128))
    for _ in range(3):
        out = tree_linear_bwd(*args, workspace=ws)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(10):
        out = tree_linear_bwd(*args, workspace=ws)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / 10
    print(f"\nlinear bwd segment tree: {ms:.3f} ms, {t.n_tokens / ms / 1e3:.1f} M tokens/s")
    assert all(torch.isfinite(o.float()).all() for o in out)


@pytest.mark.parametrize("bad", [0.0, -0.5, 1.5, float("nan")])
def test_decay_outside_unit_interval_is_reported(bad):
    """A decay outside (0, 1] lives on the device, so the host cannot refuse it:
    the forward and the backward record TREE_ATTN_ERR_INVALID_DECAY (-12) in the
    device status word instead of returning silent NaNs; the next call with a
    valid decay runs clean."""
    t = WT.Tree("decay", [-1, 0], [150, 60])
    x = WX.draw_inputs(t.n_tokens, WX.HeadConfig(2, 2, 128), WX.ValueRecipe(1, 1, 1, 1, 1), 5)
    plan = TreePlan(t.parent, t.seg_len)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    scale = 1 / np.sqrt(128)
    dec = torch.tensor([0.9, bad], dtype=torch.float32, device="cuda")
    tree_linear_fwd(plan, q, k, v, dec, scale)
    assert device_status() == -12
    tree_linear_bwd(plan, q, k, v, do, dec, scale)
    assert device_status() == -12
    good = torch.tensor([0.9, 1.0], dtype=torch.float32, device="cuda")
    o = tree_linear_fwd(plan, q, k, v, good, scale)
    assert device_status() == 0
    assert torch.isfinite(o.float()).all()
