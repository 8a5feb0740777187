"""bench.py's bounded oracle sample for the long shared context: the useful
FLOPs credited to single rows and keys add up, over every row and key of a
tree, to the step's 14*d*pairs*G (CPU only)."""
import numpy as np

import bench
from oracle import plan as OP
from workloads import trees as WT


def test_row_and_key_credits_sum_to_the_step():
    for t in (WT.tiny_binary_tree(), WT.random_tree(np.random.default_rng(3), 9, [1, 2, 5, 17]),
              WT.long_context_tree(seed=5, branches=3, lo=8, hi=64, prompt=100)):
        smp = bench.RowKeySample(t, d=128, G=8)
        pairs = OP.pair_count(t.parent, t.seg_len)
        rows = sum(smp.path_len(i) for i in range(smp.N))
        keys = sum(smp.descendants(j) for j in range(smp.N))
        assert rows == pairs and keys == pairs
        assert 128 * 8 * (10 * rows + 4 * keys) == 14 * 128 * pairs * 8


def test_sample_draws_are_valid_rows_and_leaf_end_keys():
    t = WT.long_context_tree(seed=5, branches=4, lo=8, hi=64, prompt=100)
    smp = bench.RowKeySample(t, d=128, G=8)
    for _ in range(10):
        rows, keys = smp.draw()
        assert len(set(rows)) == len(rows) and all(0 <= r < smp.N for r in rows)
        for j in keys:
            assert smp.descendants(j) <= 8
