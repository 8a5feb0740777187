"""The batching calls of the C ABI (include/tree_batch.h) against the oracle,
bit for bit, on random batches of trees (CPU only)."""
import numpy as np
import pytest

from oracle import batch as OB
from prefix_tree_attention_attn_gb300 import TreePlan
from prefix_tree_attention_attn_gb300 import _binding as B
from prefix_tree_attention_attn_gb300.batch import batch_assign, batch_forest, batch_microbatches, batch_work
from workloads import trees as WT


def random_batch(seed, n_trees):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n_trees):
        t = WT.random_tree(rng, int(rng.integers(1, 10)), [1, 3, 17, 64, 130], n_roots=int(rng.integers(1, 3)))
        out.append((t.parent, t.seg_len))
    return out


@pytest.mark.parametrize("seed", range(5))
def test_work_matches_oracle_and_plan(lib, seed):
    trees = random_batch(seed, 12)
    pairs, toks = batch_work(trees)
    for k, (p, s) in enumerate(trees):
        assert pairs[k] == OB.pairs_by_walking(p, s)
        assert toks[k] == OB.tokens(s)
        assert pairs[k] == TreePlan(p, s).n_pairs


def test_work_of_workload_trees(lib):
    names = ["tiny_binary", "grpo_star", "segment_tree", "agentic_tree"]
    trees = [(WT.load_tree(n).parent, WT.load_tree(n).seg_len) for n in names]
    pairs, toks = batch_work(trees)
    for k, (p, s) in enumerate(trees):
        assert pairs[k] == TreePlan(p, s).n_pairs and toks[k] == sum(s)


@pytest.mark.parametrize("seed,R", [(0, 1), (1, 2), (2, 3), (3, 8), (4, 64)])
def test_assign_matches_oracle(lib, seed, R):
    rng = np.random.default_rng(seed)
    work = [int(x) for x in rng.integers(0, 1000, size=int(rng.integers(1, 200)))]
    work[: len(work) // 4] = [work[0]] * (len(work) // 4)   # ties
    rep, load = batch_assign(work, R)
    orep, oload = OB.lpt(work, R)
    assert rep.tolist() == orep and load.tolist() == oload


@pytest.mark.parametrize("seed", range(4))
def test_microbatches_match_oracle(lib, seed):
    trees = random_batch(100 + seed, 40)
    pairs, toks = batch_work(trees)
    rep, _ = batch_assign(pairs, 3)
    cap = int(np.percentile(toks, 70)) * 2
    for r in range(3):
        mb, n = batch_microbatches(pairs, toks, rep, r, cap)
        omb, on = OB.microbatches(pairs.tolist(), toks.tolist(), rep.tolist(), r, cap)
        assert mb.tolist() == omb and n == on
        for m in range(n):   # the cap holds except for a tree alone above it
            members = [k for k in range(len(trees)) if mb[k] == m]
            assert sum(toks[k] for k in members) <= cap or len(members) == 1


def test_forest_matches_oracle_and_plans(lib):
    trees = random_batch(7, 9)
    sel = [k % 3 != 1 for k in range(len(trees))]
    par, seg, src = batch_forest(trees, sel)
    opar, oseg, osrc = OB.forest(trees, sel)
    assert par.tolist() == opar and seg.tolist() == oseg and src.tolist() == osrc
    # one plan over the forest: its pairs are the selected trees' pairs
    pairs, _ = batch_work(trees)
    assert TreePlan(par, seg).n_pairs == sum(int(pairs[k]) for k in range(len(trees)) if sel[k])


def test_errors(lib):
    import ctypes as C
    bad = [([-1, 0], [3, 0])]
    with pytest.raises(B.TreeAttnError) as e:
        batch_work(bad)
    assert e.value.status == -2
    with pytest.raises(B.TreeAttnError) as e:
        batch_work([([1, 0], [2, 2])])   # cycle
    assert e.value.status == -2
    with pytest.raises(B.TreeAttnError) as e:
        batch_assign([1, 2], 0)
    assert e.value.status == -1
    with pytest.raises(B.TreeAttnError) as e:
        batch_assign([1, -2], 2)
    assert e.value.status == -1
    ptr = np.array([1, 2], dtype=np.int32)    # must start at 0
    par = np.array([-1], dtype=np.int32)
    assert lib.tree_attn_batch_work(1, ptr.ctypes.data_as(B.c_int32_p), par.ctypes.data_as(B.c_int32_p),
                                    par.ctypes.data_as(B.c_int32_p), None, None) == -1
