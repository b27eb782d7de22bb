"""Pins of the oracle's balanced routing ("Outrageously Large Neural Networks -
中文验证版", section 方法适配: a per-batch mask gives every expert the same
batch size in training; per-expert thresholds approximate it at inference).

Pinned against independent routines and against the already pinned forward:
- batchwise mask: every expert keeps exactly floor(k*T/n) tokens, the same set
  as numpy's stable argsort of the column (descending score, lower token first);
- weights: torch's softmax over each token's kept experts;
- y: the dense mixture sum_e W[:, e] E_e(x) with torch's linear layers;
- thresholds at the (m+1)-th largest score of each column reproduce the
  batchwise mask; a threshold of -inf keeps every expert, which is the k = n
  layer of the oracle forward; +inf keeps none (y = 0).
"""
import numpy as np
import pytest
import torch

import oracle


def make(T, d, h, n, seed, noise=True):
    rng = np.random.default_rng(seed)
    return dict(
        x=rng.normal(size=(T, d)), Wg=rng.normal(size=(d, n)) / np.sqrt(d),
        Wn=rng.normal(size=(d, n)) / np.sqrt(d), bg=rng.normal(size=n) * 0.3,
        eps=rng.normal(size=(T, n)) if noise else None,
        W1=rng.normal(size=(n, h, d)) / np.sqrt(d), b1=rng.normal(size=(n, h)) * 0.1,
        W2=rng.normal(size=(n, d, h)) / np.sqrt(h), b2=rng.normal(size=(n, d)) * 0.1)


def scores(p):
    _, _, H, _ = oracle.gate_flat(p["x"], p["Wg"], p["Wn"], p["bg"], p["eps"], 1)
    return H


def run(p, k, thr=None):
    return oracle.forward_balanced(p["x"], p["Wg"], p["Wn"], p["bg"], p["eps"], thr, p["W1"],
                                   p["b1"], p["W2"], p["b2"], k)


def dense_mixture(p, W):
    x = torch.from_numpy(p["x"])
    y = torch.zeros_like(x)
    for e in range(p["W1"].shape[0]):
        a = torch.relu(torch.nn.functional.linear(x, torch.from_numpy(p["W1"][e]),
                                                  torch.from_numpy(p["b1"][e])))
        E = torch.nn.functional.linear(a, torch.from_numpy(p["W2"][e]), torch.from_numpy(p["b2"][e]))
        y += torch.from_numpy(W[:, e:e + 1]) * E
    return y.numpy()


@pytest.mark.parametrize("T,n,k,seed", [(40, 6, 2, 1), (37, 8, 3, 2), (64, 5, 1, 3)])
def test_batchwise_mask_weights_and_output(T, n, k, seed):
    p = make(T, 8, 12, n, seed)
    out = run(p, k)
    H = scores(p)
    m = k * T // n
    assert (out["counts"] == m).all()
    keep = out["W"] > 0
    for e in range(n):
        order = np.argsort(-H[:, e], kind="stable")     # descending, lower token first
        assert set(np.nonzero(keep[:, e])[0]) == set(order[:m].tolist())
    Ht = torch.from_numpy(H).masked_fill(torch.from_numpy(~keep), float("-inf"))
    ref_w = torch.softmax(Ht, dim=1).nan_to_num(0.0).numpy()   # rows with no kept expert -> 0
    np.testing.assert_allclose(out["W"], ref_w, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(out["y"], dense_mixture(p, out["W"]), rtol=1e-10, atol=1e-12)


def test_thresholds_at_the_batch_quantile_reproduce_the_batchwise_mask():
    T, n, k = 50, 7, 2
    p = make(T, 8, 8, n, 4)
    H = scores(p)
    m = k * T // n
    thr = -np.sort(-H, axis=0)[m]          # the (m+1)-th largest score of each column
    a, b = run(p, k), run(p, k, thr)
    np.testing.assert_array_equal(a["counts"], b["counts"])
    np.testing.assert_allclose(a["W"], b["W"], rtol=0, atol=0)
    np.testing.assert_allclose(a["y"], b["y"], rtol=0, atol=0)


def test_no_threshold_is_the_dense_layer_and_infinite_is_empty():
    T, n = 30, 5
    p = make(T, 8, 8, n, 5)
    every = run(p, 2, np.full(n, -np.inf))
    assert (every["counts"] == T).all()
    ref = oracle.forward(p["x"], p["Wg"], p["Wn"], p["bg"], p["eps"], p["W1"], p["b1"], p["W2"],
                         p["b2"], n)                       # k = n: softmax over all experts
    np.testing.assert_allclose(every["y"], ref["y"], rtol=1e-12, atol=1e-12)
    none = run(p, 2, np.full(n, np.inf))
    assert not none["counts"].any() and not none["W"].any() and not none["y"].any()


def test_noise_off_uses_the_clean_scores():
    T, n, k = 40, 6, 2
    p = make(T, 8, 8, n, 6, noise=False)
    out = run(p, k)
    c = p["x"] @ p["Wg"] + p["bg"]
    m = k * T // n
    for e in range(n):
        order = np.argsort(-c[:, e], kind="stable")
        assert set(np.nonzero(out["W"][:, e] > 0)[0]) == set(order[:m].tolist())
