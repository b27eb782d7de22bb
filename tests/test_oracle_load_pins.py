"""Pins of the oracle's load estimate (the smooth per-expert load that the load
loss balances; "Outrageously Large Neural Networks - 中文验证版", section
方法适配, with the estimate taken from the paper's load-balancing appendix).

P(t, i) is the probability that expert i stays among the k best when only its
own noise is redrawn.  The tests check it against that definition directly
(a Monte Carlo redraw with numpy), against the k = n case (every expert is
always kept) and against the vanishing-noise limit (P becomes the hard top-k
selection of the clean scores).
"""
import numpy as np
import pytest

import oracle


def _case(seed, T, d, n, scale_n=1.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    Wg = rng.standard_normal((d, n)) / np.sqrt(d)
    Wn = scale_n * rng.standard_normal((d, n)) / np.sqrt(d)
    bg = 0.3 * rng.standard_normal(n)
    eps = rng.standard_normal((T, n))
    return x, Wg, Wn, bg, eps


@pytest.mark.parametrize("n,k", [(5, 2), (6, 1), (7, 3)])
def test_load_probability_matches_monte_carlo_redraw(n, k):
    T, d = 3, 6
    x, Wg, Wn, bg, eps = _case(100 + n * 10 + k, T, d, n)
    P, load, _ = oracle.load(x, Wg, Wn, bg, eps, k)
    # definition, with library routines only
    c = x @ Wg + bg
    s = np.logaddexp(0.0, x @ Wn)
    H = c + eps * s
    rng = np.random.default_rng(7)
    N = 200_000
    for t in range(T):
        for i in range(n):
            others = np.delete(H[t], i)
            kth = np.sort(others)[::-1][k - 1]
            draws = c[t, i] + rng.standard_normal(N) * s[t, i]
            freq = float(np.mean(draws > kth))
            sigma = max(np.sqrt(freq * (1 - freq) / N), 1.0 / N)
            assert abs(freq - P[t, i]) <= 5 * sigma + 1e-4, (t, i, freq, P[t, i])
    np.testing.assert_allclose(load, P.sum(axis=0), rtol=1e-12)


def test_load_is_one_everywhere_when_k_equals_n():
    x, Wg, Wn, bg, eps = _case(3, 5, 4, 6)
    P, load, cv2 = oracle.load(x, Wg, Wn, bg, eps, 6)
    assert np.all(P == 1.0)
    np.testing.assert_array_equal(load, np.full(6, 5.0))
    assert cv2 == 0.0


def test_vanishing_noise_gives_the_hard_selection():
    # W_noise scaled so that softplus(x.W_noise) ~ e^-50: P is 0 or 1, and 1
    # exactly for the experts the (clean) gate keeps.
    T, d, n, k = 6, 8, 7, 2
    x, Wg, Wn, bg, eps = _case(4, T, d, n)
    Wn = np.full((d, n), -50.0 / d) / np.maximum(np.abs(x).mean(), 1e-9)
    Wn = -np.abs(Wn)
    x = np.abs(x)  # keeps x . W_noise strongly negative for every column
    P, _, _ = oracle.load(x, Wg, Wn, bg, eps, k)
    idx, _, _, _ = oracle.gate_flat(x, Wg, Wn, bg, None, k)  # eps None: clean scores
    hard = np.zeros((T, n))
    for t in range(T):
        hard[t, idx[t]] = 1.0
    np.testing.assert_allclose(P, hard, atol=1e-9)


def test_load_cv2_closed_form():
    x, Wg, Wn, bg, eps = _case(5, 9, 6, 5)
    _, load, cv2 = oracle.load(x, Wg, Wn, bg, eps, 2)
    assert cv2 == pytest.approx(load.var() / load.mean() ** 2, rel=1e-12)
