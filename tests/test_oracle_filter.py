"""Pins of the oracle's top-k / top-p Gumbel sampler (the issue's named
follow-up, "rejection-based top-k/top-p" on Gumbel-max; "Softmax-free GPU
sampling", Background). Reading: the filter set K is the top_k largest logits
and/or the smallest prefix (by logit) whose softmax mass reaches top_p; the
draw is the Gumbel-max over K with the same noise.

Pinned against: the unfiltered sampler when no filter is active, greedy argmax
for top_k = 1, a brute-force recomputation of K (numpy lexsort and cumulative
sums) and of the restricted argmax, the rejection identity (an unrestricted
winner that lies in K is the answer), chi-square of 1e6 draws against softmax
truncated to K, and K's support.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from tests import oracle_pool
from tests.stats_util import P_THRESHOLD, chi_square


def _k_set(x, T, top_k, top_p):
    """K by brute force: candidates ordered by (logit desc, index asc), then the
    prefix cut by top_k and by the nucleus."""
    x = np.asarray(x, dtype=np.float64)
    cand = np.flatnonzero(~(np.isnan(x) | np.isneginf(x)))
    if cand.size == 0:
        return cand
    order = cand[np.lexsort((cand, -x[cand]))]
    n = order.size
    r_k = top_k if 1 <= top_k < n else n
    r_p = n
    if top_p <= 0:
        r_p = 1
    elif top_p < 1:
        xs = x[order]
        if np.isposinf(xs).any():
            mass = np.isposinf(xs).astype(np.float64)
        else:
            mass = np.exp((xs - xs.max()) / np.float64(np.float32(T)))
        cum = np.cumsum(mass)
        r_p = int(np.argmax(cum >= np.float64(np.float32(top_p)) * cum[-1])) + 1
    return order[:min(r_k, r_p)]


def _scores(x, T, seed, row, off):
    x = np.asarray(x, dtype=np.float64)
    g = oracle.gumbel_of_words(oracle.stream_words(seed, row, off, 0, x.size))
    s = x / np.float64(np.float32(T)) + g
    s[np.isposinf(x)] = np.inf
    return s


def test_no_filter_equals_plain_sampler():
    rng = np.random.default_rng(1)
    for k in range(100):
        x = (rng.standard_normal(int(rng.integers(1, 300))) * 3).astype(np.float32)
        x[rng.random(x.size) < 0.1] = -np.inf
        for top_k, top_p in ((0, 1.0), (-3, 2.0), (10**6, float("nan"))):
            a = oracle.filtered_sample_row(x, 0.9, 11, 2, k, top_k=top_k, top_p=top_p)
            b = oracle.sample_row(x, 0.9, 11, 2, k)
            assert a[0] == b[0] and a[1] == b[1] and a[2] == np.inf


def test_top_k_one_and_top_p_zero_are_greedy():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((40, 200)) * 2).astype(np.float32)
    x[3, 5] = x[3, 17] = 50.0  # a tie: the lower index is the top element
    g, _ = oracle.argmax(x)
    for b in range(40):
        assert oracle.filtered_sample_row(x[b], 1.3, 4, b, 9, top_k=1)[0] == g[b]
        assert oracle.filtered_sample_row(x[b], 1.3, 4, b, 9, top_p=0.0)[0] == g[b]
    assert g[3] == 5


@pytest.mark.parametrize("top_k,top_p", [(3, 1.0), (0, 0.5), (0, 0.9), (7, 0.8), (40, 0.99),
                                         (1, 0.3), (2, -1.0)])
def test_brute_force_restricted_argmax(top_k, top_p):
    rng = np.random.default_rng([top_k, int(top_p * 100) & 0xFF])
    for k in range(150):
        V = int(rng.integers(1, 80))
        x = (rng.standard_normal(V) * rng.choice([0.5, 2.0, 6.0])).astype(np.float32)
        x[rng.random(V) < 0.1] = -np.inf
        x[rng.random(V) < 0.03] = np.nan
        if k % 5 == 0 and V > 2:
            x[rng.integers(0, V)] = x[rng.integers(0, V)]  # exact ties
        T = float(rng.choice([0.4, 1.0, 2.5]))
        seed, row, off = int(rng.integers(0, 2**62)), int(rng.integers(0, 64)), k
        idx, gap, _ = oracle.filtered_sample_row(x, T, seed, row, off, top_k=top_k, top_p=top_p)
        K = _k_set(x, T, top_k, top_p)
        if K.size == 0:
            assert idx == -1
            continue
        s = _scores(x, T, seed, row, off)
        sk = s[K]
        best = sk.max()
        want = int(K[sk == best].min())
        assert idx == want, (k, idx, want)
        others = np.sort(sk)[::-1]
        want_gap = np.inf if K.size == 1 else (0.0 if others[0] == others[1]
                                               else others[0] - others[1])
        assert gap == pytest.approx(want_gap, rel=0, abs=1e-12)


def test_rejection_identity():
    """When the unrestricted Gumbel-max winner lies in K it is the answer; when
    it does not, the answer is the best-scored element of K."""
    rng = np.random.default_rng(3)
    kept = rejected = 0
    for k in range(300):
        x = (rng.standard_normal(120) * 3).astype(np.float32)
        top_k, top_p = int(rng.integers(1, 30)), float(rng.uniform(0.2, 1.0))
        w, _, _ = oracle.sample_row(x, 1.0, 9, 1, k)
        f, _, _ = oracle.filtered_sample_row(x, 1.0, 9, 1, k, top_k=top_k, top_p=top_p)
        K = _k_set(x, 1.0, top_k, top_p)
        if w in K:
            kept += 1
            assert f == w
        else:
            rejected += 1
            s = _scores(x, 1.0, 9, 1, k)
            assert f in K and s[f] == s[K].max()
    assert kept > 50 and rejected > 50


def test_plus_inf_rows_and_empty_rows():
    x = np.array([1.0, np.inf, 3.0, np.inf, 2.0], np.float32)
    for top_k, top_p in ((1, 1.0), (0, 0.3), (3, 0.9)):
        assert oracle.filtered_sample_row(x, 1.0, 1, 0, 0, top_k=top_k, top_p=top_p)[0] == 1
    y = np.full(10, -np.inf, np.float32)
    assert oracle.filtered_sample_row(y, 1.0, 1, 0, 0, top_k=3, top_p=0.5)[0] == -1


def test_edge_margin_at_an_exact_boundary():
    """Two equal logits carry half the mass each; with the second one scoring
    higher, top_p = 0.5 keeps only the first and sits exactly where the second
    would join and win (margin 0); top_p = 0.75 keeps both and the winner would
    leave K only below 0.5 (margin 0.25)."""
    x = np.array([0.0, 0.0], np.float32)
    s = _scores(x, 1.0, 1, 0, 0)
    assert s[1] > s[0]  # this stream's second element wins the pair
    _, _, e = oracle.filtered_sample_row(x, 1.0, 1, 0, 0, top_p=0.5)
    assert e == 0.0
    _, _, e = oracle.filtered_sample_row(x, 1.0, 1, 0, 0, top_p=0.75)
    assert e == pytest.approx(0.25, abs=1e-7)
    # top_k binding strictly before the nucleus boundary: the margin is inactive
    x = np.zeros(10, np.float32)
    _, _, e = oracle.filtered_sample_row(x, 1.0, 1, 0, 0, top_k=2, top_p=0.9)
    assert e == np.inf


def test_edge_margin_brute_force():
    """The margin is the distance (as a share of the row's mass) from top_p to
    the nearest cut of the ordered candidates whose prefix has a different
    Gumbel-max, found here by trying every prefix length up to top_k."""
    rng = np.random.default_rng(13)
    checked = 0
    for k in range(300):
        V = int(rng.integers(2, 60))
        x = (rng.standard_normal(V) * rng.choice([0.3, 1.0, 3.0])).astype(np.float32)
        x[rng.random(V) < 0.1] = -np.inf
        T = float(rng.choice([0.5, 1.0, 2.0]))
        top_p = float(np.float32(rng.uniform(0.05, 0.98)))
        top_k = int(rng.choice([0, 3, 10, 40]))
        idx, _, e = oracle.filtered_sample_row(x, T, 21, 3, k, top_k=top_k, top_p=top_p)
        xd = x.astype(np.float64)
        cand = np.flatnonzero(~np.isneginf(xd))
        if cand.size == 0:
            continue
        order = cand[np.lexsort((cand, -xd[cand]))]
        mass = np.exp((xd[order] - xd[order].max()) / np.float64(np.float32(T)))
        S = mass.sum()
        cum = np.concatenate([[0.0], np.cumsum(mass)])  # cum[r] = mass of the first r
        n = order.size
        r_k = top_k if 1 <= top_k < n else n
        r_p = int(np.argmax(cum[1:] >= top_p * S)) + 1
        if r_k < r_p:
            assert e == np.inf
            continue
        s = _scores(x, T, 21, 3, k)[order]

        def winner(r):
            sk = s[:r]
            return int(order[:r][sk == sk.max()].min())

        assert winner(r_p) == idx
        margins = [np.inf]
        for r in range(1, r_k + 1):
            if winner(r) != idx:
                margins.append((cum[r - 1] - top_p * S) / S if r > r_p else (top_p * S - cum[r]) / S)
        assert e == pytest.approx(min(margins), rel=1e-9, abs=1e-12), (k, e, min(margins))
        checked += 1
    assert checked > 200


N_DRAWS = 1_000_000


@pytest.mark.parametrize("T", [0.5, 1.5])
@pytest.mark.parametrize("top_k,top_p", [(3, 1.0), (0, 0.8), (5, 0.9)])
def test_chi_square_against_truncated_softmax(T, top_k, top_p):
    tiny = W.tiny_statistical()
    draws = oracle_pool.filtered_steps(tiny.logits, T, 1234, 0, N_DRAWS, dtype=W.F32,
                                       top_k=top_k, top_p=top_p)
    for b in range(tiny.B):
        x = tiny.logits[b]
        K = _k_set(x, T, top_k, top_p)
        d = draws[:, b]
        assert np.isin(d, K).all(), "a draw outside the filter set"
        if K.size == 1:  # a one-element filter set: every draw is that element
            assert (d == K[0]).all()
            continue
        p = np.zeros(x.size)
        xk = x[K].astype(np.float64)
        p[K] = np.exp((xk - xk.max()) / np.float64(np.float32(T)))
        p /= p.sum()
        pval, df = chi_square(d, p)
        assert pval >= P_THRESHOLD, (b, T, top_k, top_p, pval, df)
