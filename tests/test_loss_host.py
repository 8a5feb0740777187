"""Host exports of include/tree_loss.h (trajectories, multiplicities,
position ids) against the oracle, exactly (CPU only)."""
import numpy as np
import pytest

from oracle import layout as OL
from oracle import loss as OLS
from prefix_tree_attention_attn_gb300 import TreePlan
from prefix_tree_attention_attn_gb300.loss import token_info, trajectories, trajectory_info
from workloads import trees as WT


def cases():
    rng = np.random.default_rng(11)
    out = [WT.load_tree(n) for n in ("tiny_binary", "grpo_star", "segment_tree", "agentic_tree")]
    for _ in range(8):
        out.append(WT.random_tree(rng, int(rng.integers(1, 12)), [1, 2, 7, 130], n_roots=int(rng.integers(1, 3))))
    return out


@pytest.mark.parametrize("k", range(12))
def test_trajectories_and_token_info(lib, k):
    t = cases()[k]
    plan = TreePlan(t.parent, t.seg_len)
    leaves, ptr, tok = trajectories(plan)
    ref = OL.trajectories(t.parent, t.seg_len)
    assert leaves.tolist() == [leaf for leaf, _ in ref]
    assert ptr.tolist() == np.concatenate([[0], np.cumsum([len(i) for _, i in ref])]).tolist()
    assert tok.tolist() == np.concatenate([i for _, i in ref]).tolist()
    assert trajectory_info(plan) == (len(ref), t.n_expanded)
    mult, pos = token_info(plan)
    assert mult.tolist() == OL.multiplicity(t.parent, t.seg_len).tolist()
    assert pos.tolist() == OLS.position_ids(t.parent, t.seg_len).tolist()
