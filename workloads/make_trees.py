"""Freeze the seeded workload trees as JSON fixtures under workloads/trees/.

Run from the repository root:  python -m workloads.make_trees
"""
import os

from .trees import GENERATORS, TREE_DIR


def main():
    os.makedirs(TREE_DIR, exist_ok=True)
    for name, gen in GENERATORS.items():
        t = gen()
        with open(os.path.join(TREE_DIR, name + ".json"), "w") as f:
            f.write(t.to_json() + "\n")
        print(f"{name:14s} nodes={t.n_nodes:5d} N={t.n_tokens:7d} "
              f"expanded={t.n_expanded:8d} ratio={t.n_expanded / t.n_tokens:.2f} "
              f"leaves={len(t.leaves())}")


if __name__ == "__main__":
    main()
