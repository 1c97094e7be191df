"""Writes skewed_expert_histogram.txt: how many of the 10240 tokens of the
long skewed-prefill workload (seed 3) choose each expert under the oracle's
routing.  Run from the repository root:

    python tests/golden/make_skewed_histogram.py

It calls only the input generator (``workloads``) and the oracle."""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import workloads as W  # noqa: E402
from oracle import moe_oracle as O  # noqa: E402


def main():
    li = W.skewed()
    _, idx, _ = O.route(O.bf16_bits_to_f64(li.x), li.wr, li.k)
    counts = np.bincount(idx.ravel(), minlength=li.E)
    target = np.asarray(li.notes["target_fraction"]) * li.T
    lines = [
        "# Tokens per expert of the long skewed-prefill workload (T=10240, H=2048,",
        "# E=128, top-8, seed 3) under the oracle's routing, written by",
        "# make_skewed_histogram.py.  Rows are in popularity-rank order (rank 1",
        "# first); the 16 dead experts follow with rank 0.  Columns: rank | expert |",
        "# tokens | water-filled Zipf(1.1) target T * min(1, c r^-1.1).",
    ]
    for r, e in enumerate(li.notes["rank_order"], start=1):
        lines.append(f"{r} | {e} | {counts[e]} | {target[r - 1]:.2f}")
    for e in li.notes["dead_experts"]:
        lines.append(f"0 | {e} | {counts[e]} | 0.00")
    with open(os.path.join(HERE, "skewed_expert_histogram.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
