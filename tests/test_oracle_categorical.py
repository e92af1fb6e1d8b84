"""Pins of the oracle's categorical (inverse-CDF) sampler, the baseline path of
"Softmax-free GPU sampling" (Background; Performance validation), against
closed forms and the softmax distribution rather than against itself."""
import math

import numpy as np
import pytest

import oracle
from tests.stats_util import P_THRESHOLD, chi_square, softmax64


def _u0(seed, row, offset):
    """Element 0's uniform of the row's stream (the same one the Gumbel path uses)."""
    return float(oracle.uniform_of_words(oracle.stream_words(seed, row, offset, 0, 1))[0])


def test_equal_logits_pick_floor_of_u_times_n():
    # uniform mass: the CDF steps are k/n, so the draw is floor(u * n) (closed form)
    for V in (1, 2, 7, 64):
        x = np.full(V, 0.25, np.float32)
        for off in range(200):
            idx, margin, _ = oracle.categorical_row(x, 1.0, 99, 3, off)
            u = _u0(99, 3, off)
            assert idx == min(int(math.floor(u * V)), V - 1), (V, off)
            assert 0.0 <= margin <= 0.5 / V + 1e-12


def test_masked_entries_are_skipped_in_the_cdf():
    # equal finite logits between -inf entries: the k-th finite one, k = floor(u * n)
    x = np.array([-np.inf, 1.0, -np.inf, -np.inf, 1.0, 1.0, np.nan, 1.0], np.float32)
    finite = [1, 4, 5, 7]
    for off in range(300):
        idx, _, _ = oracle.categorical_row(x, 0.7, 5, 0, off)
        assert idx == finite[int(math.floor(_u0(5, 0, off) * 4))]


def test_two_outcomes_threshold():
    # p0 = 1 / (1 + e^(d/T)); index 0 exactly when u < p0
    d, T = 1.3, float(np.float32(0.8))  # the oracle takes T as binary32
    x = np.array([0.0, d], np.float32)
    p0 = 1.0 / (1.0 + math.exp(float(x[1]) / T))
    for off in range(400):
        idx, _, _ = oracle.categorical_row(x, T, 11, 2, off)
        assert idx == (0 if _u0(11, 2, off) < p0 else 1)


@pytest.mark.parametrize("T", [0.5, 1.5])
def test_draws_follow_softmax(T):
    rng = np.random.default_rng(7)
    rows = [np.r_[rng.standard_normal(11), 4.0].astype(np.float32),     # peaked
            np.zeros(9, np.float32),                                      # flat
            np.r_[rng.standard_normal(10), 2.5, 2.5].astype(np.float32),  # bimodal
            np.r_[rng.standard_normal(8) * 2, [-np.inf] * 4].astype(np.float32)]
    n = 30000
    for x in rows:
        x = np.ascontiguousarray(x)
        draws = np.array([oracle.categorical_row(x, T, 1234, 0, k)[0] for k in range(n)])
        p = softmax64(x, T)
        assert not np.any(p[draws] == 0)  # -inf never drawn
        pv, _ = chi_square(draws, p)
        assert pv >= P_THRESHOLD, (T, pv)


def test_special_rows():
    x = np.array([1.0, 3.0, 3.0, -2.0], np.float32)
    assert oracle.categorical_row(x, 0.0, 1, 0, 0)[0] == 1           # greedy, lowest index
    assert oracle.categorical_row(x, float("nan"), 1, 0, 0)[0] == 1
    y = np.array([0.0, np.inf, 5.0, np.inf], np.float32)
    assert oracle.categorical_row(y, 1.0, 1, 0, 0)[0] == 1           # lowest +inf
    z = np.full(5, -np.inf, np.float32)
    assert oracle.categorical_row(z, 1.0, 1, 0, 0)[0] == -1          # no candidate


def test_probe_distance_locates_intervals():
    x = np.array([0.0, 0.0, 0.0, 0.0], np.float32)  # steps at 0.25, 0.5, 0.75
    for off in range(50):
        u = _u0(3, 1, off)
        idx, _, d_self = oracle.categorical_row(x, 1.0, 3, 1, off, probe=-1)
        _, _, d_hit = oracle.categorical_row(x, 1.0, 3, 1, off, probe=idx)
        assert d_hit == 0.0
        other = (idx + 2) % 4
        _, _, d_other = oracle.categorical_row(x, 1.0, 3, 1, off, probe=other)
        lo, hi = other / 4.0, (other + 1) / 4.0
        want = lo - u if u < lo else u - hi
        assert d_other == pytest.approx(want, abs=1e-12)


def test_batch_entry_matches_rows_and_bf16_input():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((5, 300)) * 2).astype(np.float32)
    T = np.array([0.5, 1.0, 0.0, 2.0, 1.0], np.float32)
    seeds = np.arange(5, dtype=np.uint64) * 77 + 1
    offs = np.arange(5, dtype=np.uint64) + 40
    idx, margin, _ = oracle.categorical(x, T, seeds, offs)
    for b in range(5):
        assert idx[b] == oracle.categorical_row(x[b], float(T[b]), int(seeds[b]), b, int(offs[b]))[0]
    # bf16 bits of values that bf16 holds exactly give the same draws
    xb = (x.view(np.uint32) & 0xFFFF0000).view(np.float32)
    bits = (xb.view(np.uint32) >> 16).astype(np.uint16)
    i32, _, _ = oracle.categorical(xb, T, seeds, offs)
    i16, _, _ = oracle.categorical(bits, T, seeds, offs, dtype=oracle.BF16)
    assert np.array_equal(i32, i16)
