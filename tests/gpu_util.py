"""Helpers shared by the GPU parity tests: run the library on seeded inputs,
compare with the fp64 oracle under the stated tolerances."""
import numpy as np
import torch

from oracle import attention as OA
from prefix_tree_attention_attn_gb300 import TreePlan, tree_attn_bwd, tree_attn_fwd

# forward: |gpu - fp64| over every element: max <= 2e-2, mean <= 2e-3
FWD_MAX, FWD_MEAN = 2e-2, 2e-3
# backward: ||g - g64||_F / ||g64||_F <= 1e-2 for dQ, dK, dV separately
BWD_REL = 1e-2


def run_gpu(t, q, k, v, do, scale, plan=None):
    plan = plan or TreePlan(t.parent, t.seg_len)
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    o, lse = tree_attn_fwd(plan, qd, kd, vd, scale)
    dq, dk, dv = tree_attn_bwd(plan, qd, kd, vd, o, lse, dod, scale)
    torch.cuda.synchronize()
    return plan, {"o": o.float().cpu().numpy(), "lse": lse.cpu().numpy().astype(np.float64),
                  "dq": dq.float().cpu().numpy(), "dk": dk.float().cpu().numpy(),
                  "dv": dv.float().cpu().numpy()}


def fwd_errors(got, ref):
    e = np.abs(got.astype(np.float64) - ref)
    return float(e.max()), float(e.mean())


def rel_fro(got, ref):
    return float(np.linalg.norm(got.astype(np.float64) - ref) / max(np.linalg.norm(ref), 1e-30))


def assert_fwd(got_o, got_lse, ref_o, ref_lse, tag=""):
    for name, g, r in (("O", got_o, ref_o), ("LSE", got_lse, ref_lse)):
        mx, mean = fwd_errors(g, r)
        assert np.isfinite(g).all(), f"{tag} {name} not finite"
        assert mx <= FWD_MAX and mean <= FWD_MEAN, f"{tag} {name}: max {mx:.3e} mean {mean:.3e}"


def assert_bwd(got, ref, tag=""):
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert np.isfinite(g).all(), f"{tag} {name} not finite"
        e = rel_fro(g, r)
        assert e <= BWD_REL, f"{tag} {name}: rel fro {e:.3e}"


def full_parity(t, q, k, v, do, scale, tag=""):
    plan, g = run_gpu(t, q, k, v, do, scale)
    ro, rl = OA.forward(t.parent, t.seg_len, q, k, v, scale)
    assert_fwd(g["o"], g["lse"], ro, rl, tag)
    rg = OA.backward(t.parent, t.seg_len, q, k, v, do, scale)
    assert_bwd((g["dq"], g["dk"], g["dv"]), rg, tag)
    return plan, g
