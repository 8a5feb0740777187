"""Full-size parity on the two largest workload trees (GPU).

Element-wise, every row and key:

* the agentic tree in full (all 32 q-heads on the GPU), with kv-group 0
  (q-heads 0-3, kv-head 0) compared with the fp64 oracle on every token:
  O, LSE and dQ of its q-heads, dK and dV of its kv-head -- the deep shared
  turns' keys included;
* a reduced long shared context: the same 32,768-token root with the first 4
  branches of the long-context recipe (seed 5), one q-head and one kv-head, so
  that the backward runs as on the full tree (q-range chunks of 64 q-tiles,
  every root kv-tile split over several items and its partial dK/dV slots
  summed in a fixed order), and again with chunks of 32 q-tiles (more than
  3,000 partial slots); every token's O, LSE, dQ, dK and dV -- the root's
  32,768 keys included, each summed over hundreds of descendant q-tiles -- is
  compared with the oracle.

For the full trees, beyond those:

The whole fp64 expansion is too expensive at these sizes (the long shared
context expands to 2.5M tokens), so the oracle checks outputs it can compute
one by one, exactly:

* O and LSE of sampled rows (each row's softmax over its own root-to-node
  path), all heads;
* dQ of the same rows (dQ_i depends on row i's path only);
* dK, dV of sampled keys near the end of leaf segments (few descendants);

and, for everything else, properties that hold at any size:

* sum_j dV_j = sum_i sum_{h in group} dO_i^h per kv-head (softmax rows sum to 1);
* sum_j dK_j = 0 per kv-head (each row of dS sums to 0);
* head-slice bit-exactness: kv-group 0 run as its own problem gives the very
  same bits for O, LSE, dK and dV as the full run (dQ, accumulated with
  atomics, within the backward tolerance).
"""
import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import layout as OL
from prefix_tree_attention_attn_gb300 import TreePlan, device_status, tree_attn_bwd, tree_attn_fwd
from workloads import tensors as WX
from workloads import trees as WT

from .gpu_util import BWD_REL, FWD_MAX, FWD_MEAN, rel_fro

pytestmark = pytest.mark.gpu


def sample_rows(t, rng, n):
    _, off, N = OL.packed_layout(t.parent, t.seg_len)
    leaves = OL.leaves(t.parent)
    rows = set(int(x) for x in rng.choice(N, size=n // 2, replace=False))
    for u in rng.choice(t.n_nodes, size=min(t.n_nodes, n // 4), replace=False):   # segment starts / ends
        rows.add(int(off[u]))
        rows.add(int(off[u] + t.seg_len[u] - 1))
    for l in leaves[:4]:
        rows.add(int(off[l] + t.seg_len[l] - 1))
    rows.update({0, N - 1, min(N - 1, 127), min(N - 1, 128)})
    return np.array(sorted(rows))


def sample_leaf_keys(t, rng, n):
    _, off, _ = OL.packed_layout(t.parent, t.seg_len)
    leaves = OL.leaves(t.parent)
    keys = []
    for l in rng.choice(leaves, size=min(len(leaves), n), replace=False):
        end = int(off[l] + t.seg_len[l])
        keys.append(end - 1 - int(rng.integers(0, min(8, t.seg_len[l]))))
    return np.array(sorted(set(keys)))


def run(plan, q, k, v, do, scale):
    o, lse = tree_attn_fwd(plan, q, k, v, scale)
    dq, dk, dv = tree_attn_bwd(plan, q, k, v, o, lse, do, scale)
    torch.cuda.synchronize()
    assert device_status() == 0
    return o, lse, dq, dk, dv


def check_workload(name, device_gen):
    t = WT.load_tree(name)
    plan = TreePlan(t.parent, t.seg_len)
    if device_gen:
        heads, rec = WX.HEADS[name], WX.VALUE_RECIPES[name]
        x = WX.draw_inputs(t.n_tokens, heads, rec, 1000 + WX.SEEDS[name], device="cuda", chunk_rows=65536)
    else:
        heads, rec, x = WX.workload_inputs(name, t.n_tokens)
        x = {kk: vv.cuda() for kk, vv in x.items()}
    scale = rec.scale
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    o, lse, dq, dk, dv = run(plan, q, k, v, do, scale)
    rng = np.random.default_rng(42)

    # ---- sampled rows: O, LSE, dQ (all heads) ----------------------------------
    rows = sample_rows(t, rng, 48)
    qc, kc, vc, doc = (a.cpu() for a in (q, k, v, do))
    ro, rl = OA.forward_rows(t.parent, t.seg_len, qc, kc, vc, scale, rows)
    go = o[torch.as_tensor(rows, device=o.device)].float().cpu().numpy()
    gl = lse[:, torch.as_tensor(rows, device=lse.device)].cpu().numpy().astype(np.float64)
    for nm, g, r in (("O", go, ro), ("LSE", gl, rl)):
        e = np.abs(g - r)
        assert e.max() <= FWD_MAX and e.mean() <= FWD_MEAN, (name, nm, e.max(), e.mean())
    rdq = OA.backward_rows_dq(t.parent, t.seg_len, qc, kc, vc, doc, scale, rows)
    gdq = dq[torch.as_tensor(rows, device=dq.device)].float().cpu().numpy()
    assert rel_fro(gdq, rdq) <= BWD_REL, (name, "dQ rows", rel_fro(gdq, rdq))

    # ---- sampled keys near leaf ends: dK, dV (all kv-heads) ----------------------
    keys = sample_leaf_keys(t, rng, 12)
    rdk, rdv = OA.backward_keys_dkdv(t.parent, t.seg_len, qc, kc, vc, doc, scale, keys)
    kk_idx = torch.as_tensor(keys, device=dk.device)
    assert rel_fro(dk[kk_idx].float().cpu().numpy(), rdk) <= BWD_REL, (name, "dK keys")
    assert rel_fro(dv[kk_idx].float().cpu().numpy(), rdv) <= BWD_REL, (name, "dV keys")

    # ---- identities over every key (they involve the heavy shared-prefix keys) ----
    G = heads.group
    sum_dv = dv.double().sum(dim=0)                                          # [hkv, d]
    want = do.double().view(t.n_tokens, heads.hkv, G, heads.d).sum(dim=(0, 2))
    assert float((sum_dv - want).norm() / want.norm()) <= BWD_REL, (name, "sum dV")
    sum_dk = dk.double().sum(dim=0)
    scale_dk = dk.double().abs().sum(dim=0)
    assert float(sum_dk.norm() / scale_dk.norm()) <= BWD_REL, (name, "sum dK")

    # ---- head slice: kv-group 0 as its own problem ----------------------------
    sl = slice(0, G)
    q0, do0 = q[:, sl].contiguous(), do[:, sl].contiguous()
    k0, v0 = k[:, 0:1].contiguous(), v[:, 0:1].contiguous()
    o0, lse0, dq0, dk0, dv0 = run(plan, q0, k0, v0, do0, scale)
    assert torch.equal(o0, o[:, sl]), name
    assert torch.equal(lse0, lse[sl]), name
    assert torch.equal(dk0, dk[:, 0:1]), name
    assert torch.equal(dv0, dv[:, 0:1]), name
    assert rel_fro(dq0.float().cpu().numpy(), dq[:, sl].float().cpu().numpy()) <= 1e-3, name


def test_agentic_tree_full_size():
    check_workload("agentic_tree", device_gen=False)


def test_long_context_full_size():
    check_workload("long_context", device_gen=True)


def compare_all(tag, got, ref):
    """Every element: O and LSE (max, mean abs), dQ, dK, dV (relative Frobenius)."""
    out = {}
    for name in ("o", "lse"):
        e = np.abs(got[name].astype(np.float64) - ref[name])
        out[name] = (float(e.max()), float(e.mean()))
    for name in ("dq", "dk", "dv"):
        out[name] = rel_fro(got[name], ref[name])
    print(f"{tag}: O max/mean {out['o'][0]:.3e}/{out['o'][1]:.3e}, LSE max/mean "
          f"{out['lse'][0]:.3e}/{out['lse'][1]:.3e}, rel Frobenius dQ {out['dq']:.3e} dK {out['dk']:.3e} "
          f"dV {out['dv']:.3e}")
    for name in ("o", "lse"):
        assert np.isfinite(got[name]).all(), (tag, name)
        assert out[name][0] <= FWD_MAX and out[name][1] <= FWD_MEAN, (tag, name, out[name])
    for name in ("dq", "dk", "dv"):
        assert np.isfinite(got[name]).all(), (tag, name)
        assert out[name] <= BWD_REL, (tag, name, out[name])


def oracle_all(t, q, k, v, do, scale):
    ro, rl = OA.forward(t.parent, t.seg_len, q, k, v, scale)
    rq, rk, rv = OA.backward(t.parent, t.seg_len, q, k, v, do, scale)
    return {"o": ro, "lse": rl, "dq": rq, "dk": rk, "dv": rv}


def test_agentic_tree_kv_group0_every_token():
    """The whole agentic tree on the GPU; kv-group 0 against the oracle on
    every token (about 2e12 useful fp64 FLOP on the host)."""
    name = "agentic_tree"
    t = WT.load_tree(name)
    plan = TreePlan(t.parent, t.seg_len)
    heads, rec, x = WX.workload_inputs(name, t.n_tokens)
    G = heads.group
    xd = {kk: vv.cuda() for kk, vv in x.items()}
    o, lse, dq, dk, dv = run(plan, xd["q"], xd["k"], xd["v"], xd["do"], rec.scale)
    got = {"o": o[:, :G].float().cpu().numpy(), "lse": lse[:G].cpu().numpy(),
           "dq": dq[:, :G].float().cpu().numpy(), "dk": dk[:, :1].float().cpu().numpy(),
           "dv": dv[:, :1].float().cpu().numpy()}
    del xd, o, lse, dq, dk, dv
    ref = oracle_all(t, x["q"][:, :G], x["k"][:, :1], x["v"][:, :1], x["do"][:, :G], rec.scale)
    compare_all("agentic tree, kv-group 0, every token", got, ref)


def test_long_context_reduced_every_token():
    """32,768-token root + the first 4 branches of the long-context recipe, one
    head: the backward as the full tree runs it (the automatic chunk of 64
    q-tiles, every root kv-tile split) and with 32-q-tile chunks (> 3,000
    partial slots), every token compared with one oracle run."""
    t = WT.long_context_tree(seed=WX.SEEDS["long_context"], branches=4)
    rec = WX.VALUE_RECIPES["long_context"]
    x = WX.draw_inputs(t.n_tokens, WX.HeadConfig(1, 1, 128), rec, 1000 + WX.SEEDS["long_context"])
    xd = {kk: vv.cuda() for kk, vv in x.items()}
    full = WT.load_tree("long_context")
    auto_chunk = TreePlan(full.parent, full.seg_len).info["bwd_chunk_qtiles"]
    runs = []
    for chunk in (0, 32):
        plan = TreePlan(t.parent, t.seg_len, bwd_chunk_qtiles=chunk)
        if chunk == 0:
            assert plan.info["bwd_chunk_qtiles"] == auto_chunk > 24, plan.info   # the full tree's chunk
        else:
            assert plan.info["n_partial_slots"] > 3000, plan.info
        assert plan.info["n_split_kv_tiles"] >= 256          # every root kv-tile is split
        o, lse, dq, dk, dv = run(plan, xd["q"], xd["k"], xd["v"], xd["do"], rec.scale)
        runs.append((plan.info["bwd_chunk_qtiles"], plan.info["n_partial_slots"],
                     {"o": o.float().cpu().numpy(), "lse": lse.cpu().numpy(), "dq": dq.float().cpu().numpy(),
                      "dk": dk.float().cpu().numpy(), "dv": dv.float().cpu().numpy()}))
        del o, lse, dq, dk, dv
    ref = oracle_all(t, x["q"], x["k"], x["v"], x["do"], rec.scale)
    root = slice(0, t.seg_len[0])
    for chunk, slots, got in runs:
        compare_all(f"long context, root + 4 branches ({t.n_tokens} tokens), chunk {chunk}, {slots} partial "
                    f"slots, every token", got, ref)
        # the root prefix's keys on their own: the ones summed over the most q-tiles
        for name in ("dk", "dv"):
            e = rel_fro(got[name][root], ref[name][root])
            print(f"  root-prefix {name}: rel Frobenius {e:.3e}")
            assert e <= BWD_REL, (name, e)
