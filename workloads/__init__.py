"""Seeded synthetic inputs for prefix-tree attention.

This package holds the tree shapes and the tensor draws that both the fp64
oracle and the GPU path consume.  It contains none of the attention
arithmetic: a tree is a parent-pointer array plus per-node segment lengths,
and a tensor set is a bundle of bf16 draws from a seeded generator.
"""
from .trees import (  # noqa: F401
    Tree,
    WORKLOADS,
    load_tree,
    tiny_binary_tree,
    grpo_star_tree,
    segment_tree,
    agentic_tree,
    long_context_tree,
    chain_tree,
    random_tree,
    expanded_forest,
)
from .tensors import HeadConfig, draw_inputs, workload_inputs  # noqa: F401
