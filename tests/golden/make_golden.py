"""Writes the stored expected values under tests/golden/ by calling the CPU
oracle only. Run from the repository root:

    python tests/golden/make_golden.py

The files pin the oracle against accidental change: any later change to the
oracle's arithmetic must regenerate them, and the commit that does so must name
the passage of the source pages (or the reading of it) that justifies it.
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import workloads as W  # noqa: E402

STEPS = 256


def tiny_draws():
    b = W.tiny_statistical()
    lines = ["# tiny_statistical workload (B=4, V=64 f32, seed 1234 every row)",
             "# columns: T step row0 row1 row2 row3  (offset = step)"]
    for T in (0.5, 1.0, 1.5):
        idx = oracle.gumbel_argmax_steps(b.logits, T, 1234, 0, STEPS)
        for k in range(STEPS):
            lines.append("%g %d %s" % (T, k, " ".join(str(int(v)) for v in idx[k])))
    return lines


def hlg_small():
    b = W.hlg(B=4, V=4096)
    p = b.hlg
    lines = ["# hlg workload recipe at B=4, V=4096 (m=1.3 w=2 beta_t=1 beta_h=1.5 c=6, T=1)",
             "# columns: pivot_mode step row0 row1 row2 row3  (offset = step)"]
    for mode in (oracle.PIVOT_TOP, oracle.PIVOT_ENTROPY):
        for k in range(64):
            idx, _ = oracle.hlg_gumbel_argmax(b.logits, b.temperature, b.seed, k, p["m"], p["w"],
                                              p["beta_t"], p["beta_h"], p["c"], mode)
            lines.append("%d %d %s" % (mode, k, " ".join(str(int(v)) for v in idx)))
    return lines


def main():
    with open(os.path.join(HERE, "oracle_tiny_draws.txt"), "w") as f:
        f.write("\n".join(tiny_draws()) + "\n")
    with open(os.path.join(HERE, "oracle_hlg_small.txt"), "w") as f:
        f.write("\n".join(hlg_small()) + "\n")


if __name__ == "__main__":
    main()
