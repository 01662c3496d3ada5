"""fp64 oracle of the Quantile-Balancing (QB) selection-bias update.

TEST INFRASTRUCTURE ONLY (tests, the smoke check and the benchmark's CPU leg).

Source: the K3 report review, section on Quantile Balancing.  For a step of m
tokens, n experts and top-k routing the target load per expert is q = m k / n.
Each token's threshold alpha_i is the (k+1)-th largest biased router score.
Expert j's new bias is the value that lets exactly q tokens' scores cross
their thresholds, i.e. a per-expert quantile of the margins; the bias only
selects and never enters the mixture weights.  At scale the quantile is
estimated from a 1000-bin histogram, with an error bounded by the bin width.

Readings (the pages print no formula for these steps):
- the router score is the sigmoid of the logit, and the bias is added to it
  (the same reading as the forward's selection key);
- the margin of token i for expert j is m_ij = alpha_i - s_ij: with bias b_j
  the token selects j exactly when s_ij + b_j > alpha_i, i.e. b_j > m_ij;
- q is rounded to the nearest integer r and kept in [1, m - 1];
- the exact update is the midpoint of the r-th and (r+1)-th smallest margins
  of the expert (any value between them makes exactly r margins cross);
- the histogram estimate spans the batch's smallest to largest margin with
  equal-width bins, and returns the upper edge of the bin holding the r-th
  smallest margin of the expert.
"""
from __future__ import annotations

import numpy as np


def scores(logits: np.ndarray) -> np.ndarray:
    """Router scores s = sigmoid(l), fp64."""
    l = np.asarray(logits, np.float64)
    return 1.0 / (1.0 + np.exp(-l))


def target_rank(m: int, n: int, k: int) -> int:
    """r = round(m k / n), kept in [1, m - 1]."""
    return int(min(max(int(np.floor(m * k / n + 0.5)), 1), m - 1))


def thresholds(s: np.ndarray, bias: np.ndarray, k: int) -> np.ndarray:
    """alpha_i: the (k+1)-th largest of s_ij + b_j over the experts j."""
    keys = s + np.asarray(bias, np.float64)[None, :]
    return np.sort(keys, axis=1)[:, -(k + 1)]


def margins(s: np.ndarray, bias: np.ndarray, k: int) -> np.ndarray:
    """m_ij = alpha_i - s_ij."""
    return thresholds(s, bias, k)[:, None] - s


def bias_exact(logits: np.ndarray, bias: np.ndarray, k: int) -> np.ndarray:
    """The exact update: midpoint of each expert's r-th and (r+1)-th smallest margin."""
    s = scores(logits)
    m, n = s.shape
    r = target_rank(m, n, k)
    srt = np.sort(margins(s, bias, k), axis=0)
    return 0.5 * (srt[r - 1] + srt[r])


def rth_margin(logits: np.ndarray, bias: np.ndarray, k: int) -> np.ndarray:
    """Each expert's r-th smallest margin (the quantile the histogram estimates)."""
    s = scores(logits)
    m, n = s.shape
    r = target_rank(m, n, k)
    return np.sort(margins(s, bias, k), axis=0)[r - 1]


def bias_histogram(logits: np.ndarray, bias: np.ndarray, k: int, nbins: int = 1000):
    """The histogram estimate; returns (bias [n], bin width)."""
    s = scores(logits)
    m, n = s.shape
    r = target_rank(m, n, k)
    mg = margins(s, bias, k)
    lo, hi = float(mg.min()), float(mg.max())
    w = (hi - lo) / nbins if hi > lo else 1.0
    b = np.clip(np.floor((mg - lo) / w).astype(np.int64), 0, nbins - 1)
    out = np.empty(n)
    for j in range(n):
        cum = np.cumsum(np.bincount(b[:, j], minlength=nbins))
        out[j] = lo + (int(np.searchsorted(cum, r)) + 1) * w
    return out, w
