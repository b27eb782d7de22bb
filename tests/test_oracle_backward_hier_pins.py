"""Pins of the oracle's backward pass for the hierarchical gate
(oracle.backward_hier).

As for the flat layer, the pages print no gradient formula: the backward is
pinned to central finite differences of the loss
L = sum_t <dy_t, y_t> + w_imp * CV^2(importance) evaluated with the oracle's
FORWARD pass of the two-level layer ("MoE:稀疏门控混合专家", section 三; the C
forward, pinned on its own).  The selection is piecewise constant, so every
case checks that no perturbation comes near a group or an in-group top-k
boundary (gate margin) and steps well inside it.  Also pinned: the shift
invariance of both softmaxes (the gate bias gradients of the group columns
sum to zero, and so do those of each group's own columns), noise off (no
gradient reaches W_noise), k_groups = 1 with one expert per group (weights
of 1 at both levels pass no gradient to the gate), and agreement with the
flat backward when there is a single group.
"""
import numpy as np
import pytest

import oracle

STEP = 1e-5


def make(T, d, h, n, groups, seed, bias=True, noise=True):
    rng = np.random.default_rng(seed)
    C = groups + n
    p = dict(
        x=rng.normal(size=(T, d)),
        Wg=rng.normal(size=(d, C)) / np.sqrt(d),
        Wn=rng.normal(size=(d, C)) / np.sqrt(d),
        bg=rng.normal(size=C) * 0.2 if bias else None,
        eps=rng.normal(size=(T, C)) if noise else None,
        W1=rng.normal(size=(n, h, d)) / np.sqrt(d),
        b1=rng.normal(size=(n, h)) * 0.1 if bias else None,
        W2=rng.normal(size=(n, d, h)) / np.sqrt(h),
        b2=rng.normal(size=(n, d)) * 0.1 if bias else None,
    )
    return p, rng.normal(size=(T, d))


def loss(p, dy, k, groups, kg, w_imp):
    f = oracle.forward(p["x"], p["Wg"], p["Wn"], p["bg"], p["eps"], p["W1"], p["b1"], p["W2"],
                       p["b2"], k, groups, kg)
    return float((dy * f["y"]).sum() + w_imp * f["cv2"]), f


def min_margin(p, k, groups, kg):
    _, _, margin = oracle.gate_hier(p["x"], p["Wg"], p["Wn"], p["bg"], p["eps"], groups, kg, k)
    return float(margin.min())


def fd_check(p, dy, k, groups, kg, w_imp, picks=6, seed=0):
    rng = np.random.default_rng(seed)
    g = oracle.backward_hier(p["x"], p["Wg"], p["Wn"], p["bg"], p["eps"], p["W1"], p["b1"],
                             p["W2"], p["b2"], dy, k, groups, kg, w_imp)
    L0, f = loss(p, dy, k, groups, kg, w_imp)
    np.testing.assert_array_equal(g["idx"], f["idx"])
    np.testing.assert_allclose(g["G"], f["G"], rtol=0, atol=1e-15)
    n = p["W1"].shape[0]
    used_e = np.unique(f["idx"])
    used_cols = np.concatenate([np.unique(f["idx"] // (n // groups)), groups + used_e])
    checked = 0
    for name in ("x", "Wg", "Wn", "bg", "W1", "b1", "W2", "b2"):
        if p[name] is None:
            continue
        arr = p[name]
        grad = g["d" + name]
        for _ in range(picks):
            i = list(np.unravel_index(rng.integers(arr.size), arr.shape))
            if name in ("W1", "b1", "W2", "b2") and rng.random() < 0.5:
                i[0] = int(rng.choice(used_e))
            if name in ("Wg", "Wn", "bg") and rng.random() < 0.7:
                i[-1] = int(rng.choice(used_cols))
            i = tuple(i)
            old = arr[i]
            arr[i] = old + STEP
            Lp, fp = loss(p, dy, k, groups, kg, w_imp)
            arr[i] = old - STEP
            Lm, fm = loss(p, dy, k, groups, kg, w_imp)
            arr[i] = old
            np.testing.assert_array_equal(fp["idx"], f["idx"])
            np.testing.assert_array_equal(fm["idx"], f["idx"])
            fd = (Lp - Lm) / (2 * STEP)
            assert abs(fd - grad[i]) <= 1e-6 * (1.0 + abs(fd)), (name, i, fd, grad[i])
            checked += 1
    return g, checked


CASES = [
    dict(T=6, d=8, h=10, n=8, groups=4, kg=2, k=4, seed=11, w_imp=0.7),
    dict(T=7, d=6, h=8, n=12, groups=3, kg=2, k=2, seed=12, w_imp=1.1),     # one expert per kept group
    dict(T=5, d=8, h=8, n=8, groups=2, kg=1, k=2, seed=13, w_imp=0.0, bias=False),
    dict(T=6, d=8, h=10, n=8, groups=4, kg=2, k=4, seed=14, w_imp=0.4, noise=False),
    dict(T=6, d=6, h=8, n=9, groups=3, kg=3, k=6, seed=15, w_imp=0.9),      # every group kept
]


@pytest.mark.parametrize("c", CASES, ids=lambda c: f"n{c['n']}_G{c['groups']}_kg{c['kg']}_k{c['k']}")
def test_backward_hier_matches_finite_differences(c):
    c = dict(c)
    w_imp, kg, k, G = c.pop("w_imp"), c.pop("kg"), c.pop("k"), c["groups"]
    bias = c.pop("bias", True)
    noise = c.pop("noise", True)
    p, dy = make(bias=bias, noise=noise, **c)
    assert min_margin(p, k, G, kg) > 1e-3
    g, checked = fd_check(p, dy, k, G, kg, w_imp, seed=c["seed"])
    assert checked >= 30
    n = c["n"]
    m = n // G
    if bias:
        scale = 1 + np.abs(g["dbg"]).sum()
        assert abs(g["dbg"][:G].sum()) < 1e-10 * scale       # group softmax
        for grp in range(G):                                    # each group's own softmax
            assert abs(g["dbg"][G + grp * m:G + (grp + 1) * m].sum()) < 1e-10 * scale
    if not noise:
        assert not g["dWn"].any()


def test_one_expert_per_group_and_one_group_pass_nothing_to_the_gate():
    p, dy = make(T=6, d=8, h=8, n=4, groups=4, seed=16)
    assert min_margin(p, 1, 4, 1) > 1e-3
    g = oracle.backward_hier(p["x"], p["Wg"], p["Wn"], p["bg"], p["eps"], p["W1"], p["b1"],
                             p["W2"], p["b2"], dy, 1, 4, 1, 0.0)
    assert np.abs(g["dWg"]).max() < 1e-12 and np.abs(g["dWn"]).max() < 1e-12
    assert np.abs(g["dbg"]).max() < 1e-12


def test_single_group_reduces_to_the_flat_backward():
    """One group holding every expert: the group weight is 1 (no gradient to
    its column) and the inner level is the flat layer over the n columns."""
    T, d, h, n, k = 6, 8, 10, 6, 2
    p, dy = make(T=T, d=d, h=h, n=n, groups=1, seed=17)
    g = oracle.backward_hier(p["x"], p["Wg"], p["Wn"], p["bg"], p["eps"], p["W1"], p["b1"],
                             p["W2"], p["b2"], dy, k, 1, 1, 0.6)
    f = oracle.backward(p["x"], p["Wg"][:, 1:], p["Wn"][:, 1:], p["bg"][1:], p["eps"][:, 1:],
                        p["W1"], p["b1"], p["W2"], p["b2"], dy, k, 0.6)
    np.testing.assert_array_equal(g["idx"], f["idx"])
    for key in ("dx", "dW1", "db1", "dW2", "db2"):
        np.testing.assert_allclose(g[key], f[key], rtol=1e-10, atol=1e-12, err_msg=key)
    np.testing.assert_allclose(g["dWg"][:, 1:], f["dWg"], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dWn"][:, 1:], f["dWn"], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dbg"][1:], f["dbg"], rtol=1e-10, atol=1e-12)
    assert np.abs(g["dWg"][:, 0]).max() < 1e-12 and abs(g["dbg"][0]) < 1e-12
