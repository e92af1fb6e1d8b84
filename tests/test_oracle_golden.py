"""The oracle still reproduces the stored draws written by
tests/golden/make_golden.py (an oracle-only script)."""
import os

import numpy as np

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_tiny_draws_golden():
    b = W.tiny_statistical()
    rows = _rows("oracle_tiny_draws.txt")
    by_T = {}
    for r in rows:
        by_T.setdefault(float(r[0]), []).append([int(v) for v in r[2:]])
    for T, want in by_T.items():
        got = oracle.gumbel_argmax_steps(b.logits, T, 1234, 0, len(want))
        assert np.array_equal(got, np.array(want)), T


def test_hlg_golden():
    b = W.hlg(B=4, V=4096)
    p = b.hlg
    for r in _rows("oracle_hlg_small.txt"):
        mode, k = int(r[0]), int(r[1])
        idx, _ = oracle.hlg_gumbel_argmax(b.logits, b.temperature, b.seed, k, p["m"], p["w"],
                                          p["beta_t"], p["beta_h"], p["c"], mode)
        assert idx.tolist() == [int(v) for v in r[2:]]
