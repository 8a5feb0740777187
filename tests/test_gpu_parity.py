"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, on
seeded inputs, element by element (forward: max / mean abs error; backward:
relative Frobenius error per tensor)."""
import numpy as np
import pytest
import torch

from prefix_tree_attention_attn_gb300 import TreePlan, device_status, tree_attn_bwd, tree_attn_fwd
from workloads import tensors as WX
from workloads import trees as WT

from .gpu_util import assert_bwd, assert_fwd, full_parity, run_gpu

pytestmark = pytest.mark.gpu


def draw(N, hq, hkv, d, seed, qk_std=1.0, do_std=1.0):
    rec = WX.ValueRecipe(qk_std, qk_std, 1.0, do_std, 1.0)
    x = WX.draw_inputs(N, WX.HeadConfig(hq, hkv, d), rec, seed)
    return x["q"], x["k"], x["v"], x["do"]


@pytest.fixture(autouse=True)
def _lib(lib, cuda_device):
    yield
    assert device_status() == 0


# --------------------------------------------------------------------------
# small cases: several tiles, ragged tails, every head layout
# --------------------------------------------------------------------------

SMALL = [
    # (parent, seg_len, hq, hkv, d)
    ([-1], [1], 2, 2, 64),                                   # one token
    ([-1], [200], 2, 1, 128),                                # single chain, ragged tail
    ([-1, 0, 0], [127, 129, 1], 4, 2, 128),                  # adversarial lengths
    ([-1, 0, 0, 1, 1], [128, 128, 255, 1, 129], 8, 2, 128),  # group 4
    ([-1, 0, 1, -1, 3], [70, 60, 5, 300, 2], 3, 3, 64),      # forest, group 1 (odd)
    ([-1, 0, 0, 0, 0, 0], [256, 40, 1, 129, 300, 7], 6, 2, 64),  # group 3 (odd)
    # caterpillar: a spine of 150 one-token nodes, each with a one-token leaf,
    # so every tile is partial and the visible keys change from row to row
    ([-1] + [2 * ((k - 1) // 2) for k in range(1, 300)], [1] * 300, 4, 2, 128),
    # wide star: a 5-token root and 300 one-token leaves (each row sees the root
    # and itself only)
    ([-1] + [0] * 300, [5] + [1] * 300, 2, 1, 64),
]


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_small_trees(case):
    parent, seg_len, hq, hkv, d = SMALL[case]
    t = WT.Tree("small", parent, seg_len)
    q, k, v, do = draw(t.n_tokens, hq, hkv, d, seed=case)
    full_parity(t, q, k, v, do, 1 / np.sqrt(d), tag=f"case{case}")


@pytest.mark.parametrize("seed", range(4))
def test_random_trees(seed):
    rng = np.random.default_rng(77 + seed)
    t = WT.random_tree(rng, int(rng.integers(3, 14)), [1, 17, 64, 127, 128, 129, 255, 300],
                       n_roots=1 + seed % 2)
    hq, hkv, d = [(4, 4, 128), (8, 2, 128), (4, 2, 64), (2, 1, 128)][seed]
    q, k, v, do = draw(t.n_tokens, hq, hkv, d, seed=100 + seed)
    full_parity(t, q, k, v, do, 1 / np.sqrt(d), tag=f"seed{seed}")


@pytest.mark.parametrize("heads", [(4, 2, 128), (3, 1, 128), (4, 2, 64), (3, 1, 64), (16, 2, 128)])
def test_long_kv_lists(heads):
    """A tree whose q-tiles see more than 24 kv-tiles on average: the forward
    then runs its long-list shapes (two q-heads per CTA for an even group size,
    one q-head per CTA with a deep ring for an odd one) instead of the
    two-CTAs-per-SM shape the other cases use."""
    t = WT.Tree("long_lists", [-1, 0, 0], [6400, 700, 900])
    plan = TreePlan(t.parent, t.seg_len)
    ex = plan.export(("qt_ptr",))
    assert (len(ex["qt_ptr"]) - 1) * 24 < ex["qt_ptr"][-1]
    hq, hkv, d = heads
    q, k, v, do = draw(t.n_tokens, hq, hkv, d, seed=31 + hq)
    full_parity(t, q, k, v, do, 1 / np.sqrt(d), tag=f"long_lists_{hq}_{hkv}")


def test_forward_kv_major_order():
    """A tree whose q-tiles stream more than 64 MB of K and V over all kv-heads
    (mean kv-tile list x 128 keys x 16 kv-heads x d = 128 x 4 bytes): the
    forward then takes its CTAs kv-head group by kv-head group.  O and LSE of
    sampled rows (every head) against the oracle, and every kv-head group run
    as its own one-kv-head problem (q-tile-major order there) gives the same
    bits."""
    from oracle import attention as OA
    t = WT.Tree("kv_major", [-1] + [0] * 8, [14000] + [600] * 8)
    plan = TreePlan(t.parent, t.seg_len)
    hq, hkv, d = 32, 16, 128
    stream = plan.info["n_tile_entries"] / plan.info["n_qtiles"] * 128 * hkv * d * 4
    assert stream > 64 * 2**20, stream
    q, k, v, _ = draw(t.n_tokens, hq, hkv, d, seed=57)
    scale = 1 / np.sqrt(d)
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o, lse = tree_attn_fwd(plan, qd, kd, vd, scale)
    G = hq // hkv
    for g in range(hkv):
        sl = slice(g * G, (g + 1) * G)
        og, lg = tree_attn_fwd(plan, qd[:, sl].contiguous(), kd[:, g:g + 1].contiguous(),
                               vd[:, g:g + 1].contiguous(), scale)
        assert torch.equal(og, o[:, sl]) and torch.equal(lg, lse[sl]), g
    rows = np.unique(np.concatenate([np.arange(0, t.n_tokens, 997), [127, 128, 14000, 14599, 14600,
                                                                      t.n_tokens - 1]]))
    ro, rl = OA.forward_rows(t.parent, t.seg_len, q, k, v, scale, rows)
    ri = torch.as_tensor(rows, device=dev)
    assert_fwd(o[ri].float().cpu().numpy(), lse[:, ri].cpu().numpy().astype(np.float64), ro, rl, tag="kv_major")


def test_sharp_logits():
    """Unscaled N(0,1) q/k with a large softmax scale: peaked rows, which
    exercise the O rescaling when the running maximum jumps."""
    t = WT.Tree("sharp", [-1, 0, 0], [300, 200, 260])
    q, k, v, do = draw(t.n_tokens, 4, 2, 128, seed=9)
    full_parity(t, q, k, v, do, 0.35, tag="sharp")


# --------------------------------------------------------------------------
# the workload trees
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny_binary", "tiny_binary_sharp"])
def test_tiny_binary_tree(name):
    t = WT.load_tree("tiny_binary")
    heads, rec, x = WX.workload_inputs(name, t.n_tokens)
    full_parity(t, x["q"], x["k"], x["v"], x["do"], rec.scale, tag=name)


@pytest.mark.parametrize("name", ["grpo_star", "segment_tree"])
def test_medium_workloads_full(name):
    t = WT.load_tree(name)
    heads, rec, x = WX.workload_inputs(name, t.n_tokens)
    full_parity(t, x["q"], x["k"], x["v"], x["do"], rec.scale, tag=name)


def test_backward_dk_dv_bitwise_reproducible():
    t = WT.load_tree("segment_tree")
    heads, rec, x = WX.workload_inputs("segment_tree", t.n_tokens)
    plan = TreePlan(t.parent, t.seg_len)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = tree_attn_fwd(plan, q, k, v, rec.scale)
    o2, lse2 = tree_attn_fwd(plan, q, k, v, rec.scale)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    _, dk1, dv1 = tree_attn_bwd(plan, q, k, v, o, lse, do, rec.scale)
    _, dk2, dv2 = tree_attn_bwd(plan, q, k, v, o, lse, do, rec.scale)
    torch.cuda.synchronize()
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)


@pytest.mark.parametrize("order", [1, 2])
def test_backward_cta_orders(order):
    """Both backward CTA orders against the oracle (the automatic rule picks
    head-major only for chunks with over 192 MB of dQ rows, i.e. the long
    context), on trees whose kv-tiles split over several chunks and several
    kv-heads; dK and dV are the same bits in either order."""
    t = WT.Tree("orders", [-1, 0, 0, 1, 2], [900, 300, 500, 129, 200])
    hq, hkv, d = 8, 2, 128
    q, k, v, do = draw(t.n_tokens, hq, hkv, d, seed=41)
    scale = 1 / np.sqrt(d)
    plan = TreePlan(t.parent, t.seg_len, bwd_chunk_qtiles=4, bwd_cta_order=order)
    assert plan.info["n_split_kv_tiles"] > 0
    _, g = run_gpu(t, q, k, v, do, scale, plan=plan)
    from oracle import attention as OA
    rg = OA.backward(t.parent, t.seg_len, q, k, v, do, scale)
    assert_bwd((g["dq"], g["dk"], g["dv"]), rg, f"order {order}")
    other = TreePlan(t.parent, t.seg_len, bwd_chunk_qtiles=4, bwd_cta_order=3 - order)
    _, g2 = run_gpu(t, q, k, v, do, scale, plan=other)
    assert np.array_equal(g["dk"], g2["dk"]) and np.array_equal(g["dv"], g2["dv"])


def test_d64_persistent_backward_walks_several_units():
    # 150 tiny binary trees as one forest: 600 (item, kv-head) units for about
    # one persistent CTA per SM, so every CTA walks several units (second K/V
    # buffer, steps counted across units, the next unit's first products while
    # the last one's dK and dV are stored)
    from prefix_tree_attention_attn_gb300 import batch as TB
    tiny = WT.load_tree("tiny_binary")
    fpar, fseg, _ = TB.TreeBatch([(tiny.parent, tiny.seg_len)] * 150).forest([True] * 150)
    t = WT.Tree("forest", [int(x) for x in fpar], [int(x) for x in fseg])
    q, k, v, do = draw(t.n_tokens, 4, 2, 64, seed=77)
    plan, _ = full_parity(t, q, k, v, do, 1 / np.sqrt(64), tag="d64 forest")
    units = plan.info["n_bwd_items"] * 2
    assert units >= 2 * torch.cuda.get_device_properties(0).multi_processor_count


def test_d64_backward_with_split_items():
    """head_dim 64 with short chunks, so kv-tiles split over several items and
    the fixed-order partial sum runs at d = 64 too."""
    t = WT.Tree("d64split", [-1, 0, 0, 2], [700, 260, 400, 300])
    hq, hkv, d = 4, 2, 64
    q, k, v, do = draw(t.n_tokens, hq, hkv, d, seed=43)
    scale = 1 / np.sqrt(d)
    plan = TreePlan(t.parent, t.seg_len, bwd_chunk_qtiles=2)
    assert plan.info["n_split_kv_tiles"] > 0 and plan.info["n_partial_slots"] > 0
    _, g = run_gpu(t, q, k, v, do, scale, plan=plan)
    from oracle import attention as OA
    ro, rl = OA.forward(t.parent, t.seg_len, q, k, v, scale)
    assert_fwd(g["o"], g["lse"], ro, rl, "d64 split")
    assert_bwd((g["dq"], g["dk"], g["dv"]), OA.backward(t.parent, t.seg_len, q, k, v, do, scale), "d64 split")
