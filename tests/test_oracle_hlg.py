"""Pins of the oracle's HLG tone curve, pivot and HLG sampler against closed
forms, library routines and the pages' own neutrality gates.

Source: "HLG sampling -- a piecewise tone curve on the logits" (mlx-bun
docs/design/hlg-sampling.md): "The transfer function" (curve and its stated
properties: C1 at the knots, slope m*beta/(beta+d) a distance d past a knot,
monotone, -inf safe), "The degeneracies are the safety anchors" (w -> inf gives
m*z; m = 1 then gives the plain sampler), "The pivot" (top: l_max - c;
entropy: sum p l), "Greedy is untouched", "Correctness & evaluation" 1-2.
"""
import math

import numpy as np
import pytest
from scipy.special import logsumexp

import oracle
import workloads as W
from tests import oracle_pool
from tests.stats_util import P_THRESHOLD, chi_square

P = W.HLG_PARAMS
M, WID, BT, BH = P["m"], P["w"], P["beta_t"], P["beta_h"]


def g(z, m=M, w=WID, bt=BT, bh=BH):
    return oracle.hlg_curve(z, m, w, bt, bh)


def test_curve_continuity_and_knot_values():
    assert g(WID)[0] == pytest.approx(M * WID, abs=1e-15)
    assert g(-WID)[0] == pytest.approx(-M * WID, abs=1e-15)
    for eps in (1e-6, 1e-9):
        assert abs(g(WID + eps)[0] - M * WID) < 2 * M * eps
        assert abs(g(-WID - eps)[0] + M * WID) < 2 * M * eps
    assert g(0.0)[0] == 0.0


def test_curve_is_c1_at_both_knots():
    h = 1e-6
    for knot in (WID, -WID):
        left = (g(knot)[0] - g(knot - h)[0]) / h
        right = (g(knot + h)[0] - g(knot)[0]) / h
        assert left == pytest.approx(M, rel=1e-5)
        assert right == pytest.approx(M, rel=1e-5)


@pytest.mark.parametrize("d", [0.25, 1.0, 3.0, 10.0])
def test_slope_decay_past_each_knot(d):
    """Slope m*beta/(beta + d) at distance d past a knot, with the shoulder's
    beta above +w and the toe's beta below -w (beta_t != beta_h here, so a
    swapped pair fails)."""
    h = 1e-5
    z = WID + d
    slope = (g(z + h)[0] - g(z - h)[0]) / (2 * h)
    assert slope == pytest.approx(M * BH / (BH + d), rel=1e-6)
    z = -WID - d
    slope = (g(z + h)[0] - g(z - h)[0]) / (2 * h)
    assert slope == pytest.approx(M * BT / (BT + d), rel=1e-6)


def test_curve_strictly_increasing_and_inf_safe():
    z = np.sort(np.random.default_rng(0).uniform(-60, 60, 1_000_000))
    z = np.unique(z)
    gz = g(z)
    assert np.all(np.diff(gz) > 0)
    ends = g(np.array([-np.inf, np.inf]))
    assert ends[0] == -np.inf and ends[1] == np.inf
    assert not np.any(np.isnan(ends))


def test_rolloff_off_is_linear_gain():
    z = np.random.default_rng(1).uniform(-40, 40, 10000)
    assert np.array_equal(oracle.hlg_curve(z, 1.7, np.inf, BT, BH), 1.7 * z)
    assert np.array_equal(oracle.hlg_curve(z, 1.0, np.inf, BT, BH), z)


def test_odd_symmetry_when_betas_match():
    z = np.random.default_rng(2).uniform(0, 30, 1000)
    assert np.allclose(oracle.hlg_curve(-z, 1.3, 2.0, 1.5, 1.5), -oracle.hlg_curve(z, 1.3, 2.0, 1.5, 1.5),
                       rtol=0, atol=1e-12)


def _row(seed=3, V=4096, inf_frac=0.01):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal(V) * 3).astype(np.float32)
    x[rng.random(V) < inf_frac] = -np.inf
    return x


def test_pivot_top_against_library_logsumexp():
    x = _row()
    lse, mu = oracle.hlg_pivot(x, c=6.0)
    fin = x[np.isfinite(x)].astype(np.float64)
    assert lse == pytest.approx(logsumexp(fin), rel=0, abs=1e-12)
    assert mu == pytest.approx((fin.max() - logsumexp(fin)) - 6.0, abs=1e-12)
    # the most probable token sits exactly c nats above the pivot: z_max = c
    t = oracle.hlg_transform_row(x, 1.0, np.inf, 1.0, 1.0, 6.0)
    assert t[np.nanargmax(np.where(np.isfinite(x), x, -np.inf))] == pytest.approx(6.0, abs=1e-12)


def test_pivot_entropy_closed_forms():
    for n in (1, 2, 7, 1000):
        x = np.zeros(n, dtype=np.float32)
        _, mu = oracle.hlg_pivot(x, c=0.0, pivot_mode=oracle.PIVOT_ENTROPY)
        assert mu == pytest.approx(-math.log(n), abs=1e-12)
    for a in (0.1, 0.5, 0.9):
        x = np.array([math.log(a), math.log(1 - a), -np.inf], dtype=np.float32)
        pa = math.exp(float(x[0])) / (math.exp(float(x[0])) + math.exp(float(x[1])))
        _, mu = oracle.hlg_pivot(x, c=0.0, pivot_mode=oracle.PIVOT_ENTROPY)
        assert mu == pytest.approx(pa * math.log(pa) + (1 - pa) * math.log(1 - pa), abs=1e-7)
    assert oracle.hlg_pivot(np.full(5, -np.inf, dtype=np.float32), c=0.0) is None


def test_transform_masks_and_ranks():
    x = _row(4)
    t = oracle.hlg_transform_row(x, M, WID, BT, BH, 6.0)
    assert np.all(np.isneginf(t[np.isneginf(x)]))
    fin = np.isfinite(x)
    order = np.argsort(x[fin], kind="stable")
    assert np.all(np.diff(t[fin][order]) >= 0)  # rank-preserving
    assert np.nanargmax(np.where(fin, t, -np.inf)) == np.nanargmax(np.where(fin, x, -np.inf))


def _plain_vs_hlg(x, T_plain, T_hlg, m, c, offsets):
    B = x.shape[0]
    seeds = W.splitmix64(11, B)
    same = 0
    for off in offsets:
        a, ga = oracle.gumbel_argmax(x, T_plain, seeds, off)
        h, gh = oracle.hlg_gumbel_argmax(x, T_hlg, seeds, off, m, np.inf, BT, BH, c)
        near = (ga < 1e-9) | (gh < 1e-9)
        assert np.all((a == h) | near)
        same += int(np.sum(a == h))
    return same


def test_neutrality_identity_config_equals_plain_sampler():
    """m = 1 with the rolloff off: HLG is the plain sampler (the pivot shift is
    a per-row constant, which the argmax ignores)."""
    x = np.stack([_row(s, V=2048) for s in range(6)])
    for T in (0.6, 1.0, 1.4):
        assert _plain_vs_hlg(x, T, T, 1.0, 6.0, range(20)) == 6 * 20


def test_neutrality_gain_folds_temperature():
    """Rolloff off with m = 1/T0 at temperature 1 equals plain temperature T0."""
    x = np.stack([_row(s, V=2048) for s in range(6)])
    for T0 in (0.5, 2.0):
        assert _plain_vs_hlg(x, T0, 1.0, 1.0 / T0, 3.0, range(20)) == 6 * 20


def test_greedy_untouched_and_plus_inf():
    x = np.stack([_row(s, V=512) for s in range(4)])
    for T in (0.0, -2.0, np.nan):
        a, _ = oracle.hlg_gumbel_argmax(x, T, 1, 1, M, WID, BT, BH, 6.0)
        r, _ = oracle.argmax(x)
        assert np.array_equal(a, r)
    y = x.copy()
    y[2, 100] = np.inf
    y[2, 300] = np.inf
    a, _ = oracle.hlg_gumbel_argmax(y, 1.0, 1, 1, M, WID, BT, BH, 6.0)
    assert a[2] == 100


def _softmax(v, T):
    q = np.where(np.isfinite(v), v / T, -np.inf)
    e = np.exp(q - q[np.isfinite(q)].max())
    return e / e.sum()


@pytest.mark.parametrize("T,mode", [(1.0, oracle.PIVOT_TOP), (0.7, oracle.PIVOT_TOP),
                                    (1.0, oracle.PIVOT_ENTROPY)])
def test_hlg_draws_follow_softmax_of_tone_mapped_logprobs(T, mode):
    """Gumbel-max over g(z)/T is an exact sample of softmax(g(z)/T)."""
    rng = np.random.default_rng(21)
    x = (rng.standard_normal(64) * 3).astype(np.float32)
    x[rng.choice(64, 6, replace=False)] = -np.inf
    params = dict(m=M, w=WID, beta_t=BT, beta_h=BH, c=6.0, pivot_mode=mode)
    draws = oracle_pool.hlg_row_steps(x, W.F32, T, 77, 0, 0, 200_000, params)
    assert not np.any(np.isneginf(x[draws]))
    tone = oracle.hlg_transform_row(x, M, WID, BT, BH, 6.0, mode)
    pval, df = chi_square(draws, _softmax(tone, T))
    assert pval >= P_THRESHOLD, (pval, df)
