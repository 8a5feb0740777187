"""fp64 CPU oracle for prefix-tree attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The library never calls it and shares no code
with it: the GPU path has its own planner (C++) and kernels (CUDA).

What it computes (the equivalence the pages require): every token of a rollout
prefix tree must get the output and gradients it would get if its root-to-leaf
trajectory were trained on its own (AReaL-DTA abstract and HARTS abstract:
separate training of each trajectory computes the shared prefixes again for
every trajectory, forward and backward).  So the oracle expands every trajectory,
runs plain dense causal softmax attention on it in fp64, and maps the results
back onto the compact tokens.

Modules:
  layout     -- packed token order, trajectories, multiplicities, ancestor sets
  attention  -- expanded-trajectory forward/backward, plus a second,
                independent compact-space masked formula
  plan       -- brute-force tile plan derived from the dense ancestor mask

Pins (tests in ``tests/test_oracle_*.py``, all CPU): a single chain equals
``torch.nn.functional.scaled_dot_product_attention(is_causal=True)`` forward
and (through autograd) backward; pure-Python brute force on every small tree;
closed forms with constant logits; central finite differences of <O, dO>;
torch autograd through the compact masked formula; invariants (copies agree,
dO split invariance, sibling permutation, chain merging, forest = separate
trees, softmax rows sum to one).
"""
