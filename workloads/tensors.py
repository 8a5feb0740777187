"""Seeded bf16 inputs (Q, K, V, dO) for a packed tree.

Tensors are token-major ``[N, H, d]`` in the packed (compact) token order;
which compact token belongs to which node is fixed by the packing convention,
not by this module.  Values are drawn in fp32 from a seeded
``torch.Generator`` in the order Q, K, V, dO, scaled, then rounded to bf16, so
the oracle and the GPU see identical bits.

Value recipes (``VALUE_RECIPES``), per workload:

* tiny binary tree: Q, K, V ~ N(0, 1) / sqrt(64); dO ~ N(0, 1); scale 1.0
  (the 1/sqrt(d) is already in the inputs).  A "sharp" variant keeps Q, K, V
  unscaled and uses scale 1/sqrt(64).
* GRPO star: Q, V ~ N(0, 1); K ~ N(0, 1) / sqrt(128); dO ~ N(0, 1e-2) read as
  variance 1e-2 (std 0.1); scale 1.0.
* segment tree: Q, K, V, dO ~ N(0, 1); scale 1/sqrt(128).
* agentic tree: Q, K, V ~ N(0, 1); dO std 0.1; scale 1/sqrt(128).
* long shared context: Q, K, V, dO ~ N(0, 1); scale 1/sqrt(128).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch


@dataclasses.dataclass(frozen=True)
class HeadConfig:
    hq: int
    hkv: int
    d: int

    @property
    def group(self) -> int:
        return self.hq // self.hkv


@dataclasses.dataclass(frozen=True)
class ValueRecipe:
    q_std: float
    k_std: float
    v_std: float
    do_std: float
    scale: float


HEADS = {
    "tiny_binary": HeadConfig(2, 2, 64),
    "grpo_star": HeadConfig(32, 8, 128),
    "segment_tree": HeadConfig(32, 8, 128),
    "agentic_tree": HeadConfig(32, 8, 128),
    "long_context": HeadConfig(64, 8, 128),
}

VALUE_RECIPES = {
    "tiny_binary": ValueRecipe(1 / 8, 1 / 8, 1 / 8, 1.0, 1.0),
    "tiny_binary_sharp": ValueRecipe(1.0, 1.0, 1.0, 1.0, 1 / 8),
    "grpo_star": ValueRecipe(1.0, 1 / math.sqrt(128), 1.0, 0.1, 1.0),
    "segment_tree": ValueRecipe(1.0, 1.0, 1.0, 1.0, 1 / math.sqrt(128)),
    "agentic_tree": ValueRecipe(1.0, 1.0, 1.0, 0.1, 1 / math.sqrt(128)),
    "long_context": ValueRecipe(1.0, 1.0, 1.0, 1.0, 1 / math.sqrt(128)),
}

SEEDS = {"tiny_binary": 1, "tiny_binary_sharp": 1, "grpo_star": 2, "segment_tree": 3,
         "agentic_tree": 4, "long_context": 5}


def draw_inputs(n_tokens: int, heads: HeadConfig, recipe: ValueRecipe, seed: int,
                device: str = "cpu", chunk_rows: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Draw Q, K, V, dO as bf16 ``[N, H, d]`` tensors.

    ``device`` selects where the generator runs (a CUDA generator draws a
    different but equally seeded stream; used only for sizes the host cannot
    hold comfortably).  ``chunk_rows`` bounds the fp32 temporaries.
    """
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = {}
    specs = [("q", heads.hq, recipe.q_std), ("k", heads.hkv, recipe.k_std),
             ("v", heads.hkv, recipe.v_std), ("do", heads.hq, recipe.do_std)]
    for name, h, std in specs:
        t = torch.empty((n_tokens, h, heads.d), dtype=torch.bfloat16, device=device)
        step = chunk_rows or max(n_tokens, 1)
        for r0 in range(0, n_tokens, step):
            r1 = min(n_tokens, r0 + step)
            x = torch.randn((r1 - r0, h, heads.d), generator=g, dtype=torch.float32, device=device)
            if std != 1.0:
                x.mul_(std)
            t[r0:r1].copy_(x)
        out[name] = t
    return out


def workload_inputs(name: str, n_tokens: int, device: str = "cpu",
                    chunk_rows: Optional[int] = None):
    """(heads, recipe, tensors) for a named workload of ``n_tokens`` tokens."""
    base = "tiny_binary" if name.startswith("tiny_binary") else name
    heads = HEADS[base]
    recipe = VALUE_RECIPES[name]
    return heads, recipe, draw_inputs(n_tokens, heads, recipe, 1000 + SEEDS[name],
                                      device=device, chunk_rows=chunk_rows)
