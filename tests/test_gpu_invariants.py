"""Invariants of the GPU path that hold whatever the oracle says (GPU).

* merging a single-child chain into one node changes nothing: the token plan
  is the same, so O, LSE, dK and dV are bit-identical (dQ, accumulated with
  atomics, to rounding);
* a forest of chains whose lengths are multiples of the 128-token tile gives
  each chain exactly what a call on that chain alone gives (same tiles, same
  order of work), again bit for bit except dQ;
* relabelling nodes so that siblings are visited in another order moves the
  tokens but gives every node the same outputs and gradients (to rounding,
  since the tile boundaries move).
"""
import numpy as np
import pytest
import torch

from oracle import layout as OL
from prefix_tree_attention_attn_gb300 import TreePlan, device_status, tree_attn_bwd, tree_attn_fwd
from workloads import tensors as WX
from workloads import trees as WT

pytestmark = pytest.mark.gpu

HEADS = WX.HeadConfig(8, 2, 128)
SCALE = 1 / np.sqrt(128)


def draw(n, seed):
    x = WX.draw_inputs(n, HEADS, WX.ValueRecipe(1, 1, 1, 1, 1), seed)
    return [x[k].cuda() for k in ("q", "k", "v", "do")]


def run(parent, seg_len, q, k, v, do):
    plan = TreePlan(parent, seg_len)
    o, lse = tree_attn_fwd(plan, q, k, v, SCALE)
    dq, dk, dv = tree_attn_bwd(plan, q, k, v, o, lse, do, SCALE)
    torch.cuda.synchronize()
    assert device_status() == 0
    return plan, (o, lse, dq, dk, dv)


def close(a, b, tol):
    a, b = a.float(), b.float()
    return float((a - b).norm() / b.norm().clamp_min(1e-30)) <= tol


def test_chain_merge_is_bit_identical(lib, cuda_device):
    q, k, v, do = draw(600, 1)
    _, a = run([-1, 0, 1, 2], [130, 200, 70, 200], q, k, v, do)
    _, b = run([-1], [600], q, k, v, do)
    for x, y in zip(a[:2] + a[3:], b[:2] + b[3:]):        # O, LSE, dK, dV
        assert torch.equal(x, y)
    assert close(a[2], b[2], 1e-5)                          # dQ


def test_forest_of_aligned_chains_equals_separate_calls(lib, cuda_device):
    lens = [256, 384, 128]
    q, k, v, do = draw(sum(lens), 2)
    _, full = run([-1] * len(lens), lens, q, k, v, do)
    start = 0
    for L in lens:
        s = slice(start, start + L)
        _, part = run([-1], [L], q[s].contiguous(), k[s].contiguous(), v[s].contiguous(), do[s].contiguous())
        o, lse, dq, dk, dv = full
        assert torch.equal(part[0], o[s])
        assert torch.equal(part[1], lse[:, s])
        assert torch.equal(part[3], dk[s])
        assert torch.equal(part[4], dv[s])
        assert close(part[2], dq[s], 1e-5)
        start += L


def test_sibling_order_does_not_matter(lib, cuda_device):
    rng = np.random.default_rng(5)
    t = WT.random_tree(rng, 9, [40, 100, 129, 200], n_roots=1)
    perm = rng.permutation(t.n_nodes)                   # old id -> new id
    p2 = [0] * t.n_nodes
    l2 = [0] * t.n_nodes
    for old in range(t.n_nodes):
        par = t.parent[old]
        p2[perm[old]] = -1 if par < 0 else int(perm[par])
        l2[perm[old]] = t.seg_len[old]
    q, k, v, do = draw(t.n_tokens, 3)
    _, off1, _ = OL.packed_layout(t.parent, t.seg_len)
    _, off2, _ = OL.packed_layout(p2, l2)
    # the same per-node values, packed in each tree's own order
    idx = torch.empty(t.n_tokens, dtype=torch.long)
    for old in range(t.n_nodes):
        L = t.seg_len[old]
        idx[off2[perm[old]]:off2[perm[old]] + L] = torch.arange(off1[old], off1[old] + L)
    ii = idx.cuda()
    _, a = run(t.parent, t.seg_len, q, k, v, do)
    _, b = run(p2, l2, q[ii].contiguous(), k[ii].contiguous(), v[ii].contiguous(), do[ii].contiguous())
    o, lse, dq, dk, dv = a
    for x, y, tol in ((b[0], o[ii], 1e-2), (b[2], dq[ii], 1e-2), (b[3], dk[ii], 1e-2), (b[4], dv[ii], 1e-2)):
        assert close(x, y, tol)
    assert float((b[1] - lse[:, ii]).abs().max()) <= 1e-2


def test_bounded_wait_timeout_is_reported_and_context_survives(lib, cuda_device):
    """A wait that nothing completes runs out after its limit, the kernel
    returns and records the timeout; the next calls work normally."""
    import prefix_tree_attention_attn_gb300._binding as B
    assert device_status() == 0
    st = B.load().tree_attn_selftest_wait_timeout(50, None)
    assert st == 0
    code = device_status()
    assert code == -10 - 1000 * 99, code
    assert B.load().tree_attn_strerror(code).decode().startswith("a bounded device wait")
    assert device_status() == 0          # read and cleared
    from .gpu_util import full_parity
    t = WT.Tree("after", [-1, 0], [130, 70])
    x = WX.draw_inputs(t.n_tokens, HEADS, WX.ValueRecipe(1, 1, 1, 1, 1), 4)
    full_parity(t, x["q"], x["k"], x["v"], x["do"], SCALE, tag="after-timeout")
    assert device_status() == 0
