"""Chi-square goodness of fit of sampled indices against exact softmax
probabilities (the regression guard of "Softmax-free GPU sampling: Gumbel-max
categorical sampling kernel": >= 1e6 draws, several logit shapes, temperatures
0.5 and 1.5, masked tokens never drawn)."""
import numpy as np
from scipy import stats

P_THRESHOLD = 1e-4  # per (row, temperature) test; 12 tests -> ~1.2e-3 family-wise


def softmax64(x: np.ndarray, T: float) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    finite = np.isfinite(x)
    q = np.where(finite, x / T, -np.inf)
    m = q[finite].max()
    e = np.where(finite, np.exp(q - m), 0.0)
    return e / e.sum()


def chi_square(draws: np.ndarray, p: np.ndarray):
    """Returns (pvalue, df). Bins with expected count < 5 are pooled."""
    n = draws.size
    counts = np.bincount(draws, minlength=p.size).astype(np.float64)
    expected = p * n
    big = expected >= 5
    obs = list(counts[big])
    exp = list(expected[big])
    small_exp = expected[~big & (p > 0)].sum()
    if small_exp > 0:
        obs.append(counts[~big & (p > 0)].sum())
        exp.append(small_exp)
    obs = np.array(obs)
    exp = np.array(exp)
    exp *= obs.sum() / exp.sum()
    res = stats.chisquare(obs, exp)
    return res.pvalue, len(obs) - 1
