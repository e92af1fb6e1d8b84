"""Pins of the oracle's uniform mapping and Gumbel transform against closed
forms (not against a retyped formula).

Reading (the pages only say "u from a counter-based stream"): u = ((r >> 9) +
0.5) * 2^-23, and g = -log(-log u) ("Softmax-free GPU sampling: Gumbel-max
categorical sampling kernel", Background).
"""
import math

import numpy as np

import oracle

EULER_GAMMA = 0.57721566490153286061


def _all_cells():
    k = np.arange(1 << 23, dtype=np.uint32)
    return k << np.uint32(9)


def test_uniform_closed_form():
    u = oracle.uniform_of_words(np.array([0, 511, 512, 0xFFFFFFFF, 0x80000000], dtype=np.uint32))
    assert u[0] == 2.0**-24 and u[1] == 2.0**-24  # low 9 bits ignored
    assert u[2] == 3 * 2.0**-24
    assert u[3] == 1 - 2.0**-24
    assert u[4] == 0.5 + 2.0**-24
    r = np.random.default_rng(1).integers(0, 2**32, 100000, dtype=np.uint64).astype(np.uint32)
    ur = oracle.uniform_of_words(r)
    un = oracle.uniform_of_words(~r)
    assert np.all(ur + un == 1.0)  # symmetric: u(r) + u(~r) = 1 exactly
    assert np.all(ur.astype(np.float32).astype(np.float64) == ur)  # exact in binary32
    assert np.all((ur > 0) & (ur < 1))


def test_gumbel_grid_moments_and_cdf():
    """Over all 2^23 equally likely cells the transform must reproduce the
    standard Gumbel law: mean = Euler's gamma, variance = pi^2/6, and
    P(g <= t) = exp(-exp(-t)). The midpoint grid errs by O(2^-23 log 2^23)."""
    g = oracle.gumbel_of_words(_all_cells())
    assert abs(g.mean() - EULER_GAMMA) < 2e-6
    assert abs(g.var() - math.pi**2 / 6) < 1e-4
    for t in (-1.5, -0.5, 0.0, 0.5, 1.0, 2.0, 4.0, 8.0):
        emp = np.mean(g <= t)
        assert abs(emp - math.exp(-math.exp(-t))) < 4 * 2.0**-23 + 1e-7, t
    # monotone in the 23 random bits, extremes at the grid ends
    assert np.all(np.diff(g) > 0)
    assert abs(g[-1] - (-math.log(-math.log1p(-2.0**-24)))) < 1e-12
    assert g[-1] < 16.6356 and g[-1] > 16.6354


def test_gumbel_point_values():
    # u = exp(-1) gives g = 0; u = exp(-exp(-t)) gives g = t (the inverse CDF)
    for t in (-2.0, 0.0, 1.0, 3.5, 10.0):
        u = math.exp(-math.exp(-t))
        assert abs(oracle.gumbel(u) - t) < 1e-9 * max(1.0, abs(t)) + 1e-12 / (1 - u + 1e-300)
