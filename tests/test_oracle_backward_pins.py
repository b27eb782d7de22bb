"""Pins of the oracle's backward pass (flat gating).

The pages train the layer but print no gradient formula, so the backward is
pinned to something other than itself: central finite differences of the loss
L = sum_t <dy_t, y_t> + w_imp * CV^2(importance) evaluated with the oracle's
FORWARD pass (pinned on its own to the pages' worked example, brute-force
top-k, the dense softmax mixture and torch's linear layers).  The selection is
piecewise constant, so every case checks that no perturbation comes near a
top-k boundary (gate margin) and steps well inside it.  Also pinned: the
softmax's shift invariance (the bias gradients of the gate sum to zero), k = 1
(a weight of 1 has no gradient to pass to the gate), noise off (no gradient
reaches W_noise) and the zero loss.
"""
import numpy as np
import pytest

import oracle

STEP = 1e-5


def make(T, d, h, n, k, seed, bias=True, noise=True):
    rng = np.random.default_rng(seed)
    p = dict(
        x=rng.normal(size=(T, d)),
        Wg=rng.normal(size=(d, n)) / np.sqrt(d),
        Wn=rng.normal(size=(d, n)) / np.sqrt(d),
        bg=rng.normal(size=n) * 0.2 if bias else None,
        eps=rng.normal(size=(T, n)) if noise else None,
        W1=rng.normal(size=(n, h, d)) / np.sqrt(d),
        b1=rng.normal(size=(n, h)) * 0.1 if bias else None,
        W2=rng.normal(size=(n, d, h)) / np.sqrt(h),
        b2=rng.normal(size=(n, d)) * 0.1 if bias else None,
    )
    dy = rng.normal(size=(T, d))
    return p, dy


def loss(p, dy, k, w_imp):
    f = oracle.forward(p["x"], p["Wg"], p["Wn"], p["bg"], p["eps"], p["W1"], p["b1"], p["W2"],
                       p["b2"], k)
    return float((dy * f["y"]).sum() + w_imp * f["cv2"]), f


def min_margin(p, k):
    idx, G, H, margin = oracle.gate_flat(p["x"], p["Wg"], p["Wn"], p["bg"], p["eps"], k)
    return float(margin.min())


def fd_check(p, dy, k, w_imp, picks=5, seed=0):
    rng = np.random.default_rng(seed)
    g = oracle.backward(p["x"], p["Wg"], p["Wn"], p["bg"], p["eps"], p["W1"], p["b1"], p["W2"],
                        p["b2"], dy, k, w_imp)
    L0, f = loss(p, dy, k, w_imp)
    np.testing.assert_array_equal(g["idx"], f["idx"])
    used = np.unique(f["idx"])
    checked = 0
    for name in ("x", "Wg", "Wn", "bg", "W1", "b1", "W2", "b2"):
        if p[name] is None:
            continue
        arr = p[name]
        grad = g["d" + name]
        for _ in range(picks):
            i = list(np.unravel_index(rng.integers(arr.size), arr.shape))
            # expert-indexed parameters: pick a routed expert half the time
            if name in ("W1", "b1", "W2", "b2") and rng.random() < 0.5:
                i[0] = int(rng.choice(used))
            if name in ("Wg", "Wn") and rng.random() < 0.5:
                i[-1] = int(rng.choice(used))
            i = tuple(i)
            old = arr[i]
            arr[i] = old + STEP
            Lp, fp = loss(p, dy, k, w_imp)
            arr[i] = old - STEP
            Lm, fm = loss(p, dy, k, w_imp)
            arr[i] = old
            np.testing.assert_array_equal(fp["idx"], f["idx"])
            np.testing.assert_array_equal(fm["idx"], f["idx"])
            fd = (Lp - Lm) / (2 * STEP)
            assert abs(fd - grad[i]) <= 1e-6 * (1.0 + abs(fd)), (name, i, fd, grad[i])
            checked += 1
    return g, checked


CASES = [
    dict(T=6, d=8, h=12, n=6, k=2, seed=1, w_imp=0.7),
    dict(T=5, d=6, h=10, n=4, k=4, seed=2, w_imp=1.3),            # dense: k = n
    dict(T=7, d=8, h=8, n=5, k=3, seed=3, w_imp=0.0, bias=False),  # no biases, no aux loss
    dict(T=6, d=8, h=12, n=6, k=2, seed=4, w_imp=0.5, noise=False),
    dict(T=8, d=6, h=8, n=7, k=1, seed=5, w_imp=0.9),
]


@pytest.mark.parametrize("c", CASES, ids=lambda c: f"T{c['T']}_n{c['n']}_k{c['k']}_s{c['seed']}")
def test_backward_matches_finite_differences(c):
    c = dict(c)
    w_imp = c.pop("w_imp")
    bias = c.pop("bias", True)
    noise = c.pop("noise", True)
    p, dy = make(bias=bias, noise=noise, **c)
    assert min_margin(p, c["k"]) > 1e-3
    g, checked = fd_check(p, dy, c["k"], w_imp, seed=c["seed"])
    assert checked >= 20
    if bias:
        # softmax shift invariance: sum over slots of dH is zero per token
        assert abs(g["dbg"].sum()) < 1e-10 * (1 + np.abs(g["dbg"]).sum())
    if not noise:
        assert not g["dWn"].any()
    if c["k"] == 1:
        # one kept expert has weight 1 whatever its score: no gate gradient
        assert np.abs(g["dWg"]).max() < 1e-12 and np.abs(g["dWn"]).max() < 1e-12


def test_importance_loss_alone():
    """dy = 0: only w_imp * CV^2 drives the gradient; it matches finite
    differences and scales linearly with w_imp."""
    p, dy = make(T=6, d=8, h=8, n=5, k=2, seed=6)
    dy[:] = 0.0
    assert min_margin(p, 2) > 1e-3
    g1, _ = fd_check(p, dy, 2, 1.0, seed=6)
    g2 = oracle.backward(p["x"], p["Wg"], p["Wn"], p["bg"], p["eps"], p["W1"], p["b1"], p["W2"],
                         p["b2"], dy, 2, 2.0)
    np.testing.assert_allclose(g2["dWg"], 2.0 * g1["dWg"], rtol=1e-12, atol=1e-15)
    assert not g1["dW1"].any() and not g1["dW2"].any()   # experts see no gradient


def test_zero_loss_gives_zero_gradients():
    p, dy = make(T=4, d=6, h=8, n=4, k=2, seed=7)
    g = oracle.backward(p["x"], p["Wg"], p["Wn"], p["bg"], p["eps"], p["W1"], p["b1"], p["W2"],
                        p["b2"], np.zeros_like(dy), 2, 0.0)
    for key in ("dx", "dWg", "dWn", "dbg", "dW1", "db1", "dW2", "db2"):
        assert not g[key].any(), key
