"""Pins of the oracle's top-two gap: the quantity that decides which sampled
rows the parity rule exempts (indices must equal the oracle's except where the
two best perturbed scores are closer than 1e-5).

The oracle keeps the best and second-best score in one streaming pass. Here the
gap is recomputed by brute force: every score of the row, a full sort, the
difference of the two largest. The scores use the oracle's Gumbel transform and
stream words, which are pinned on their own (Gumbel law over all 2^23 cells,
cuRAND's Philox), so these tests check only the bookkeeping: a best that is
replaced must become the runner-up, a later runner-up must still be seen, and
masked entries never count.

Source: "Softmax-free GPU sampling: Gumbel-max categorical sampling kernel",
Background (score = logits/T + g, one index-carrying max per row).
"""
import numpy as np
import pytest

import oracle


def _scores(x, T, seed, row_id, offset):
    """Every element's perturbed score in double; masked entries get -inf."""
    x = np.asarray(x, dtype=np.float64)
    T = float(np.float32(T))  # the oracle takes the temperature as binary32
    g = oracle.gumbel_of_words(oracle.stream_words(seed, row_id, offset, 0, x.size))
    s = x / T + g
    s[np.isinf(x) & (x > 0)] = np.inf
    s[np.isnan(x) | (np.isneginf(x))] = -np.inf
    return s


def _brute(s):
    """(index, gap) from a full sort: lowest index of the largest score, and the
    largest minus the second largest (inf with fewer than two candidates)."""
    live = s[s > -np.inf]
    if live.size == 0:
        return -1, np.inf
    idx = int(np.flatnonzero(s == live.max())[0])
    if live.size == 1:
        return idx, np.inf
    top = np.sort(live)[::-1]
    gap = 0.0 if top[0] == top[1] else float(top[0] - top[1])
    return idx, gap


@pytest.mark.parametrize("T", [0.5, 1.0, 2.0])
def test_two_element_rows(T):
    rng = np.random.default_rng(int(T * 10))
    for k in range(200):
        x = (rng.standard_normal(2) * 2).astype(np.float32)
        idx, gap, best = oracle.sample_row(x, T, 1000 + k, 3, k)
        w = oracle.stream_words(1000 + k, 3, k, 0, 2)
        g = oracle.gumbel_of_words(w)
        s0 = float(x[0]) / T + g[0]
        s1 = float(x[1]) / T + g[1]
        assert gap == abs(s0 - s1)
        assert idx == (0 if s0 >= s1 else 1)
        assert best == max(s0, s1)


def test_best_replaced_twice_demotes_the_old_best():
    """Strictly increasing scores (logits 200 apart, |g| < 17): every element
    replaces the best, so the runner-up is always the element just before."""
    x = np.array([0.0, 200.0, 400.0], np.float32)
    idx, gap, _ = oracle.sample_row(x, 1.0, 77, 0, 5)
    s = _scores(x, 1.0, 77, 0, 5)
    assert idx == 2
    assert gap == s[2] - s[1]
    # five replacements in a row
    x = np.arange(6, dtype=np.float32) * 300.0
    idx, gap, _ = oracle.sample_row(x, 1.0, 78, 1, 9)
    s = _scores(x, 1.0, 78, 1, 9)
    assert idx == 5 and gap == s[5] - s[4]


def test_runner_up_after_the_best():
    """The best comes first, the runner-up last, a low element between them."""
    x = np.array([400.0, 0.0, 200.0], np.float32)
    idx, gap, _ = oracle.sample_row(x, 1.0, 79, 2, 1)
    s = _scores(x, 1.0, 79, 2, 1)
    assert idx == 0 and gap == s[0] - s[2]
    # runner-up between two lower elements, best in the middle
    x = np.array([0.0, 300.0, 900.0, 600.0, 100.0], np.float32)
    idx, gap, _ = oracle.sample_row(x, 1.0, 80, 2, 1)
    s = _scores(x, 1.0, 80, 2, 1)
    assert idx == 2 and gap == s[2] - s[3]


def test_brute_force_on_random_rows():
    rng = np.random.default_rng(123)
    for k in range(400):
        V = int(rng.integers(1, 60))
        x = (rng.standard_normal(V) * rng.choice([0.5, 3.0, 20.0])).astype(np.float32)
        x[rng.random(V) < 0.15] = -np.inf
        x[rng.random(V) < 0.05] = np.nan
        if k % 7 == 0 and V > 3:
            x[rng.integers(0, V)] = np.inf
        T = float(rng.choice([0.3, 1.0, 4.0]))
        seed, row, off = int(rng.integers(0, 2**63)), int(rng.integers(0, 512)), k
        idx, gap, _ = oracle.sample_row(x, T, seed, row, off)
        bidx, bgap = _brute(_scores(x, T, seed, row, off))
        assert idx == bidx, (k, idx, bidx)
        assert gap == bgap, (k, gap, bgap)


def test_equal_scores_give_zero_gap():
    """Two copies of one logit with the same word are impossible within a row,
    but two +inf logits, or a flat row at a huge temperature's scale, tie."""
    x = np.array([1.0, np.inf, 3.0, np.inf], np.float32)
    idx, gap, _ = oracle.sample_row(x, 1.0, 5, 0, 0)
    assert idx == 1 and gap == 0.0


def test_batch_entry_reports_each_rows_gap():
    rng = np.random.default_rng(7)
    B, V = 6, 40
    x = (rng.standard_normal((B, V)) * 3).astype(np.float32)
    T = np.array([0.5, 1.0, 1.5, 0.7, 2.0, 1.0], np.float32)
    seeds = np.arange(B, dtype=np.uint64) * 31 + 1
    offs = np.arange(B, dtype=np.uint64) + 4
    idx, gap = oracle.gumbel_argmax(x, T, seeds, offs)
    for b in range(B):
        bidx, bgap = _brute(_scores(x[b], float(T[b]), int(seeds[b]), b, int(offs[b])))
        assert idx[b] == bidx and gap[b] == bgap


def test_greedy_gap_is_difference_of_two_largest_logits():
    rng = np.random.default_rng(8)
    for k in range(200):
        V = int(rng.integers(1, 50))
        x = rng.integers(-5, 5, V).astype(np.float32)  # small integers: many ties
        x[rng.random(V) < 0.1] = -np.inf
        idx, gap = oracle.argmax(x[None, :])
        bidx, bgap = _brute(np.where(np.isnan(x), -np.inf, x.astype(np.float64)))
        assert idx[0] == bidx and gap[0] == bgap, (k, x)


def test_hlg_gap_brute_force():
    """The HLG sampler's gap over the tone-mapped scores g(z)/T + gumbel."""
    rng = np.random.default_rng(9)
    curve = dict(m=1.3, w=2.0, beta_t=1.0, beta_h=1.5, c=6.0)
    for k in range(100):
        V = int(rng.integers(2, 80))
        x = (rng.standard_normal(V) * 3).astype(np.float32)
        x[rng.random(V) < 0.1] = -np.inf
        if not np.isfinite(x).any():
            x[0] = 0.0
        T = float(rng.choice([0.5, 1.0, 1.7]))
        mode = k % 2
        idx, gap, _ = oracle.hlg_sample_row(x, T, 11 + k, 2, k, pivot_mode=mode, **curve)
        y = oracle.hlg_transform_row(x, curve["m"], curve["w"], curve["beta_t"], curve["beta_h"],
                                     curve["c"], pivot_mode=mode)
        g = oracle.gumbel_of_words(oracle.stream_words(11 + k, 2, k, 0, V))
        s = np.where(np.isfinite(x), y / float(np.float32(T)) + g, -np.inf)
        bidx, bgap = _brute(s)
        assert idx == bidx and gap == pytest.approx(bgap, rel=0, abs=1e-12), (k, gap, bgap)
