"""Pins of the Quantile-Balancing bias oracle (oracle/qb.py) against what the
K3 report review's QB section fixes: the target load q = m k / n, the
(k+1)-th-score token threshold, exactly q crossings per expert under the new
bias, and the histogram estimate's error bounded by the bin width."""
import numpy as np

from oracle import qb


def _count_selected(logits, bias, k):
    """Tokens that select each expert under ``bias`` against the thresholds
    alpha computed with the same bias: plain comparisons, no sorting."""
    s = qb.scores(logits)
    alpha = qb.thresholds(s, bias, k)
    return (s + bias[None, :] > alpha[:, None]).sum(axis=0)


def _count_crossing(logits, old_bias, new_bias, k):
    """Tokens whose score plus the new bias beats the threshold fixed by the old bias."""
    s = qb.scores(logits)
    alpha = qb.thresholds(s, old_bias, k)
    return (s + new_bias[None, :] > alpha[:, None]).sum(axis=0)


def test_target_rank():
    assert qb.target_rank(8192, 896, 16) == 146          # 146.29
    assert qb.target_rank(32768, 896, 16) == 585         # 585.14
    assert qb.target_rank(16, 896, 16) == 1              # 0.29 -> kept at 1
    assert qb.target_rank(100, 10, 5) == 50


def test_hand_worked_case():
    # 4 tokens, 3 experts, top-1, no bias: q = 4/3 -> r = 1.
    l = np.log(np.array([[0.9, 0.5, 0.1],
                         [0.2, 0.8, 0.3],
                         [0.6, 0.7, 0.4],
                         [0.3, 0.1, 0.5]]) / (1 - np.array([[0.9, 0.5, 0.1],
                                                           [0.2, 0.8, 0.3],
                                                           [0.6, 0.7, 0.4],
                                                           [0.3, 0.1, 0.5]])))
    s = qb.scores(l)
    assert np.allclose(s[0], [0.9, 0.5, 0.1])
    # second-largest score per token
    alpha = qb.thresholds(s, np.zeros(3), 1)
    assert np.allclose(alpha, [0.5, 0.3, 0.6, 0.3])
    # margins alpha - s, per expert sorted: e0 {-0.4, 0.1, 0.0, 0.0}, e1 {0, -0.5, -0.1, 0.2},
    # e2 {0.4, 0.0, 0.2, -0.2}; midpoint of the 1st and 2nd smallest
    assert np.allclose(qb.bias_exact(l, np.zeros(3), 1), [-0.2, -0.3, -0.1])


def _count_at_or_below(logits, old_bias, new_bias, k):
    s = qb.scores(logits)
    alpha = qb.thresholds(s, old_bias, k)
    return (s + new_bias[None, :] >= alpha[:, None]).sum(axis=0)


def test_r_tokens_cross():
    # exactly r margins lie below the new bias, up to ties: every token whose
    # (k+1)-th pick is expert j itself has margin b_j (old) exactly, so the
    # statement is #{m < b} <= r <= #{m <= b}; with a zero old bias the count
    # is exactly r for every expert whose r-th margin is not in that tie group
    rng = np.random.default_rng(5)
    for m, n, k in [(512, 64, 4), (2000, 96, 8), (300, 16, 2)]:
        l = rng.standard_normal((m, n)) * 2.0
        b0 = rng.standard_normal(n) * 0.05
        nb = qb.bias_exact(l, b0, k)
        r = qb.target_rank(m, n, k)
        assert np.all(_count_crossing(l, b0, nb, k) <= r)
        assert np.all(_count_at_or_below(l, b0, nb, k) >= r)
    l = rng.standard_normal((1000, 40))
    b0 = np.zeros(40)
    nb = qb.bias_exact(l, b0, 3)
    r = qb.target_rank(1000, 40, 3)
    exact = _count_crossing(l, b0, nb, 3) == r
    ties = np.isclose(nb, 0.0)
    assert np.all(exact | ties) and exact.sum() >= 10


def test_update_balances_a_skewed_router():
    # experts with a large score offset get a negative bias, starved ones a positive one
    rng = np.random.default_rng(6)
    m, n, k = 4096, 32, 4
    l = rng.standard_normal((m, n)) + np.linspace(-1.5, 1.5, n)[None, :]
    b = np.zeros(n)
    before = _count_selected(l, b, k)
    nb = qb.bias_exact(l, b, k)
    assert np.corrcoef(np.linspace(-1.5, 1.5, n), nb)[0, 1] < -0.95
    after = _count_selected(l, nb, k)
    q = m * k / n
    assert np.abs(after - q).max() < 0.1 * np.abs(before - q).max()
    # repeated updates (the bias of one step routes the next) keep closing the gap
    dev = [np.abs(after - q).max()]
    for _ in range(4):
        nb = qb.bias_exact(l, nb, k)
        dev.append(np.abs(_count_selected(l, nb, k) - q).max())
    assert dev[-1] < dev[0]


def test_histogram_within_one_bin_of_the_quantile():
    rng = np.random.default_rng(7)
    l = rng.standard_normal((3000, 48)) * 1.5
    b0 = rng.standard_normal(48) * 0.02
    est, w = qb.bias_histogram(l, b0, 6, nbins=1000)
    exact_r = qb.rth_margin(l, b0, 6)
    d = est - exact_r
    assert np.all(d > 0) and np.all(d <= w * (1 + 1e-9))
    # finer bins -> closer
    est2, w2 = qb.bias_histogram(l, b0, 6, nbins=4000)
    assert np.abs(est2 - exact_r).max() <= w2 * (1 + 1e-9) < w
