"""Pins of the CPU oracle to facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: a value the
pages print (the worked example), a closed form, brute force over all expert
subsets, or a special case that reduces to an independent library routine
(numpy / torch CPU).  Every stage (noisy score, KeepTopK, softmax, routing,
importance, CV^2, expert FFN, combine) is covered by at least one test that a
dropped term, a wrong sign, a wrong index or a transposed operand would fail.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# --------------------------------------------------------------------------
# Worked example: "MoE:稀疏门控混合专家", section 三 (8 experts, keep 2).
# --------------------------------------------------------------------------
@pytest.mark.parametrize("fill_seed", [0, 1, 2])
def test_worked_example_of_the_gate(fill_seed):
    rows = _read_golden("worked_example_gate.txt")
    kv = {}
    scores, pexp, pw = {}, {}, {}
    for r in rows:
        if r[0] == "score":
            scores[int(r[1])] = float(r[2])
        elif r[0] == "printed_exp":
            pexp[int(r[1])] = float(r[2])
        elif r[0] == "printed_weight":
            pw[int(r[1])] = float(r[2])
        else:
            kv[r[0]] = r[1]
    n, k, dec = int(kv["n"]), int(kv["k"]), int(kv["printed_decimals"])
    # The six unprinted scores: any values below the second best.
    rng = np.random.default_rng(fill_seed)
    s = rng.uniform(-3.0, 2.0, size=n)
    for e, v in scores.items():
        s[e] = v
    d = 3
    x = np.zeros((1, d))
    x[0, 0] = 1.0                      # x = e_0, so x . W_g = row 0 of W_g
    Wg = np.zeros((d, n))
    Wg[0] = s
    Wn = np.zeros((d, n))
    idx, G, H, _ = oracle.gate_flat(x, Wg, Wn, None, None, k)
    top = sorted(scores, key=lambda e: -scores[e])
    assert idx[0].tolist() == top                         # experts 2 then 5
    np.testing.assert_allclose(H[0], s, rtol=0, atol=0)   # eps absent: H = x.W_g
    # Printed weights to the page's two decimals.
    assert [round(float(g), dec) for g in G[0]] == [pw[e] for e in top]
    # Printed e^score values reproduce the weight within their rounding (+-0.005).
    a, b = pexp[top[0]], pexp[top[1]]
    bound = (b * 0.005 + a * 0.005) / (a + b) ** 2
    assert abs(G[0, 0] - a / (a + b)) <= bound
    assert abs(G[0, 1] - b / (a + b)) <= bound
    assert round(math.exp(scores[top[0]]), dec) == a and round(math.exp(scores[top[1]]), dec) == b


# --------------------------------------------------------------------------
# softplus ("MoE:稀疏门控混合专家", section 四): closed forms and a library routine.
# --------------------------------------------------------------------------
def test_softplus_closed_forms():
    assert oracle.softplus(0.0) == pytest.approx(math.log(2.0), abs=1e-16)
    assert oracle.softplus(2.0) == pytest.approx(2.1269280110429727, abs=1e-15)  # ln(1+e^2)
    assert oracle.softplus(50.0) == pytest.approx(50.0, abs=1e-15)
    assert oracle.softplus(-50.0) == pytest.approx(math.exp(-50.0), rel=1e-12)
    assert oracle.softplus(800.0) == 800.0          # no overflow
    for z in np.linspace(-30, 30, 121):
        # softplus(z) - softplus(-z) = z
        assert oracle.softplus(z) - oracle.softplus(-z) == pytest.approx(z, abs=1e-12)
        ref = torch.nn.functional.softplus(torch.tensor(z, dtype=torch.float64),
                                           threshold=1000.0).item()
        assert oracle.softplus(z) == pytest.approx(ref, rel=1e-14, abs=1e-300)


# --------------------------------------------------------------------------
# Noisy score H = x.W_g + eps * softplus(x.W_noise), closed-form cases.
# --------------------------------------------------------------------------
def test_noise_term_closed_form():
    # d = 1, x = 1: clean score c_i = W_g[0,i], noise score r_i = W_noise[0,i].
    c = np.array([[1.0, 0.9, 0.0, 0.5]])
    r = np.array([[0.0, 2.0, -30.0, 0.0]])
    eps = np.array([[0.0, 1.0, 5.0, -1.0]])
    x = np.ones((1, 1))
    idx, G, H, _ = oracle.gate_flat(x, c, r, None, eps, 2)
    sp2 = math.log1p(math.exp(2.0))
    expect_H = [1.0, 0.9 + sp2, 5.0 * math.log1p(math.exp(-30.0)), 0.5 - math.log(2.0)]
    np.testing.assert_allclose(H[0], expect_H, rtol=1e-15, atol=1e-300)
    assert idx[0].tolist() == [1, 0]
    e1, e0 = math.exp(0.9 + sp2), math.exp(1.0)
    np.testing.assert_allclose(G[0], [e1 / (e1 + e0), e0 / (e1 + e0)], rtol=1e-14)


def test_gate_bias_added_to_clean_score():
    x = np.ones((1, 1))
    c = np.array([[0.0, 0.1, 0.2]])
    bg = np.array([0.5, 0.0, -1.0])
    idx, G, H, _ = oracle.gate_flat(x, c, np.zeros_like(c), bg, None, 1)
    np.testing.assert_allclose(H[0], [0.5, 0.1, -0.8], rtol=0, atol=1e-16)
    assert idx[0].tolist() == [0] and G[0, 0] == 1.0


def test_noise_off_reduces_to_matmul():
    rng = np.random.default_rng(7)
    x, Wg, Wn = rng.normal(size=(9, 16)), rng.normal(size=(16, 6)), rng.normal(size=(16, 6))
    _, _, H, _ = oracle.gate_flat(x, Wg, Wn, None, None, 2)
    np.testing.assert_allclose(H, x @ Wg, rtol=1e-12, atol=1e-12)
    _, _, H0, _ = oracle.gate_flat(x, Wg, Wn, None, np.zeros((9, 6)), 2)
    np.testing.assert_allclose(H0, x @ Wg, rtol=1e-12, atol=1e-12)


def test_noisy_scores_match_library_routines():
    rng = np.random.default_rng(8)
    x, Wg, Wn = rng.normal(size=(7, 12)), rng.normal(size=(12, 5)), rng.normal(size=(12, 5))
    eps = rng.normal(size=(7, 5))
    _, _, H, _ = oracle.gate_flat(x, Wg, Wn, None, eps, 2)
    sp = torch.nn.functional.softplus(torch.from_numpy(x @ Wn)).numpy()
    np.testing.assert_allclose(H, x @ Wg + eps * sp, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# KeepTopK + softmax: brute force over all C(n,k) subsets, and the library softmax.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("n,k", [(n, k) for n in range(1, 9) for k in range(1, min(n, 3) + 1)])
def test_top_k_equals_brute_force(n, k):
    rng = np.random.default_rng(100 * n + k)
    T, d = 24, 5
    x = rng.normal(size=(T, d))
    Wg, Wn = rng.normal(size=(d, n)), rng.normal(size=(d, n))
    eps = rng.normal(size=(T, n))
    idx, G, H, margin = oracle.gate_flat(x, Wg, Wn, None, eps, k)
    for t in range(T):
        best = max(itertools.combinations(range(n), k), key=lambda c: sum(H[t, list(c)]))
        assert set(idx[t].tolist()) == set(best)
        assert all(H[t, idx[t, j]] >= H[t, idx[t, j + 1]] for j in range(k - 1))
        masked = torch.full((n,), float("-inf"), dtype=torch.float64)
        masked[list(best)] = torch.from_numpy(H[t, list(best)])
        ref = torch.softmax(masked, 0).numpy()
        np.testing.assert_allclose(G[t], ref[idx[t]], rtol=1e-14, atol=1e-16)
        assert np.count_nonzero(ref) == k
        assert G[t].sum() == pytest.approx(1.0, abs=1e-15)
        assert np.all((G[t] > 0) & (G[t] <= 1))
        srt = np.sort(H[t])[::-1]
        assert margin[t] == (srt[k - 1] - srt[k] if k < n else np.inf)


def test_softmax_shift_invariance_and_ties_to_lower_index():
    x = np.ones((1, 1))
    s = np.array([[0.3, 1.0, 1.0, 0.2, 1.0]])
    idx, G, _, margin = oracle.gate_flat(x, s, np.zeros_like(s), None, None, 2)
    assert idx[0].tolist() == [1, 2] and margin[0] == 0.0
    idx2, G2, _, _ = oracle.gate_flat(x, s + 123.0, np.zeros_like(s), None, None, 2)
    assert idx2[0].tolist() == [1, 2]
    np.testing.assert_allclose(G2, G, rtol=1e-15)


# --------------------------------------------------------------------------
# Hierarchical MoE-N-h ("MoE:稀疏门控混合专家", section 三: 16 x 256, 2 then 2).
# --------------------------------------------------------------------------
def _hier_case(rng, T, G, m, noisy):
    d = 6
    C = G + G * m
    return (rng.normal(size=(T, d)), rng.normal(size=(d, C)), rng.normal(size=(d, C)),
            rng.normal(size=C) * 0.3, rng.normal(size=(T, C)) if noisy else None)


@pytest.mark.parametrize("G,m,kg,ki", [(g, m, kg, ki) for g in (1, 2, 3, 4) for m in (1, 2, 4)
                                       for kg in range(1, g + 1) for ki in range(1, m + 1)])
def test_hierarchical_equals_brute_force(G, m, kg, ki):
    rng = np.random.default_rng(1000 * G + 100 * m + 10 * kg + ki)
    T = 10
    x, Wg, Wn, bg, eps = _hier_case(rng, T, G, m, noisy=True)
    idx, Gw, _ = oracle.gate_hier(x, Wg, Wn, bg, eps, G, kg, kg * ki)
    # Scores per column via library routines, then brute-force selection per level.
    Hall = x @ Wg + bg + eps * torch.nn.functional.softplus(torch.from_numpy(x @ Wn)).numpy()
    for t in range(T):
        hp = Hall[t, :G]
        groups = max(itertools.combinations(range(G), kg), key=lambda c: sum(hp[list(c)]))
        groups = sorted(groups, key=lambda g: -hp[g])
        mp = torch.full((G,), float("-inf"), dtype=torch.float64)
        mp[groups] = torch.from_numpy(hp[groups])
        gp = torch.softmax(mp, 0).numpy()
        expect_idx, expect_w = [], []
        for g in groups:
            hi = Hall[t, G + g * m:G + (g + 1) * m]
            inner = max(itertools.combinations(range(m), ki), key=lambda c: sum(hi[list(c)]))
            inner = sorted(inner, key=lambda e: -hi[e])
            mi = torch.full((m,), float("-inf"), dtype=torch.float64)
            mi[inner] = torch.from_numpy(hi[inner])
            gi = torch.softmax(mi, 0).numpy()
            expect_idx += [g * m + e for e in inner]
            expect_w += [gp[g] * gi[e] for e in inner]
        assert idx[t].tolist() == expect_idx
        np.testing.assert_allclose(Gw[t], expect_w, rtol=1e-13, atol=1e-16)
        # exactly kg distinct groups with ki experts each; weights sum to 1
        grp = idx[t] // m
        assert len(set(grp.tolist())) == kg
        assert all((grp == g).sum() == ki for g in set(grp.tolist()))
        assert Gw[t].sum() == pytest.approx(1.0, abs=1e-14)


def test_hierarchical_single_group_reduces_to_flat():
    rng = np.random.default_rng(5)
    T, m, d = 16, 8, 6
    x = rng.normal(size=(T, d))
    Wg, Wn = rng.normal(size=(d, 1 + m)), rng.normal(size=(d, 1 + m))
    eps = rng.normal(size=(T, 1 + m))
    idx_h, G_h, _ = oracle.gate_hier(x, Wg, Wn, None, eps, 1, 1, 3)
    idx_f, G_f, _, _ = oracle.gate_flat(x, Wg[:, 1:], Wn[:, 1:], None, eps[:, 1:], 3)
    assert np.array_equal(idx_h, idx_f)
    np.testing.assert_allclose(G_h, G_f, rtol=1e-15)


def test_hierarchical_one_expert_per_group_is_the_flat_group_gate():
    """m = 1: every kept group holds one expert with in-group weight 1, so the
    layer's choice and weights are the flat gate over the G group columns."""
    rng = np.random.default_rng(6)
    T, G, d = 20, 7, 6
    x = rng.normal(size=(T, d))
    Wg, Wn = rng.normal(size=(d, 2 * G)), rng.normal(size=(d, 2 * G))
    bg, eps = rng.normal(size=2 * G) * 0.3, rng.normal(size=(T, 2 * G))
    idx_h, G_h, _ = oracle.gate_hier(x, Wg, Wn, bg, eps, G, 3, 3)
    idx_f, G_f, _, _ = oracle.gate_flat(x, Wg[:, :G], Wn[:, :G], bg[:G], eps[:, :G], 3)
    assert np.array_equal(idx_h, idx_f)
    np.testing.assert_allclose(G_h, G_f, rtol=1e-15)


@pytest.mark.parametrize("G,m,kg,ki", [(4, 6, 2, 3), (3, 5, 3, 2), (5, 4, 2, 1)])
def test_hierarchical_levels_are_flat_gates(G, m, kg, ki):
    """Each level of the two-level gate is the (independently pinned) flat
    gate on its own columns: the kept groups and the group weights (the sums
    of each group's final weights) are the flat gate over the group columns,
    and within a kept group the experts and the weight ratios are the flat
    gate over that group's columns; the final weight is their product."""
    rng = np.random.default_rng(100 * G + m)
    T = 25
    x, Wg, Wn, bg, eps = _hier_case(rng, T, G, m, noisy=True)
    idx_h, G_h, _ = oracle.gate_hier(x, Wg, Wn, bg, eps, G, kg, kg * ki)
    idx_g, G_g, _, _ = oracle.gate_flat(x, Wg[:, :G], Wn[:, :G], bg[:G], eps[:, :G], kg)
    for t in range(T):
        for q in range(kg):
            sl = slice(q * ki, (q + 1) * ki)
            g = int(idx_g[t, q])
            assert set((idx_h[t, sl] // m).tolist()) == {g}
            wsum = G_h[t, sl].sum()
            assert wsum == pytest.approx(G_g[t, q], rel=1e-13)
            cols = slice(G + g * m, G + (g + 1) * m)
            idx_i, G_i, _, _ = oracle.gate_flat(x[t:t + 1], Wg[:, cols], Wn[:, cols], bg[cols],
                                                eps[t:t + 1, cols], ki)
            assert (idx_h[t, sl] - g * m).tolist() == idx_i[0].tolist()
            np.testing.assert_allclose(G_h[t, sl] / wsum, G_i[0], rtol=1e-12)
            np.testing.assert_allclose(G_h[t, sl], G_g[t, q] * G_i[0], rtol=1e-12)


# --------------------------------------------------------------------------
# Routing: counts, offsets, stable permutation, importance, CV^2.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("T,n,k", [(0, 4, 2), (1, 1, 1), (37, 5, 2), (300, 16, 4), (64, 3, 3)])
def test_route_against_library(T, n, k):
    rng = np.random.default_rng(T * 31 + n)
    idx = np.stack([rng.permutation(n)[:k] for _ in range(T)]) if T else np.zeros((0, k), np.int32)
    G = rng.dirichlet(np.ones(k), size=T) if T else np.zeros((0, k))
    counts, offsets, perm, inv_perm, imp, cv2 = oracle.route(idx, G, n)
    flat = idx.reshape(-1)
    assert np.array_equal(counts, np.bincount(flat, minlength=n))
    assert offsets[0] == 0 and np.array_equal(offsets[1:], np.cumsum(counts))
    assert offsets[-1] == T * k and counts.sum() == T * k
    assert counts.mean() == pytest.approx(k * T / n)       # ~k*b/n rows per expert
    assert np.array_equal(perm, np.argsort(flat, kind="stable"))
    assert np.array_equal(inv_perm[perm], np.arange(T * k))
    np.testing.assert_allclose(imp, np.bincount(flat, weights=G.reshape(-1), minlength=n),
                               rtol=1e-13, atol=1e-13)
    assert imp.sum() == pytest.approx(T, rel=1e-13, abs=1e-13)
    ref = np.var(imp) / np.mean(imp) ** 2 if T else 0.0
    assert cv2 == pytest.approx(ref, rel=1e-12, abs=1e-15)


def test_cv2_closed_forms():
    n, T = 6, 12
    # every token on expert 0 (k=1): importance = [T,0,...,0], CV^2 = n - 1
    idx = np.zeros((T, 1), np.int32)
    *_, imp, cv2 = oracle.route(idx, np.ones((T, 1)), n)
    assert cv2 == pytest.approx(n - 1, rel=1e-14)
    # perfectly balanced: CV^2 = 0
    idx = (np.arange(T) % n).reshape(T, 1).astype(np.int32)
    *_, cv2 = oracle.route(idx, np.ones((T, 1)), n)
    assert cv2 == 0.0
    # two of four experts share everything equally: CV^2 = 1
    idx = (np.arange(8) % 2).reshape(8, 1).astype(np.int32)
    *_, cv2 = oracle.route(idx, np.ones((8, 1)), 4)
    assert cv2 == pytest.approx(1.0, rel=1e-14)


def test_route_rejects_bad_expert_index():
    with pytest.raises(ValueError):
        oracle.route(np.array([[0, 5]], np.int32), np.ones((1, 2)) / 2, 4)


# --------------------------------------------------------------------------
# Expert FFN and combine.
# --------------------------------------------------------------------------
def test_expert_parameter_count_matches_page():
    # "MoE:稀疏门控混合专家", section 二: 512 x 1024 + 1024 x 512 = 1048576 weights.
    from sparsely_gated_mixture_top_b300 import workloads as wl
    w = wl.WORKLOADS["flat_n256_k4"]
    W1, W2 = wl.expert_weight(w, "W1", 3), wl.expert_weight(w, "W2", 3)
    assert W1.numel() + W2.numel() == 1048576


def test_single_expert_reduces_to_plain_ffn():
    rng = np.random.default_rng(11)
    T, d, h = 20, 16, 24           # d != h: a transposed weight would fail
    x = rng.normal(size=(T, d))
    W1, W2 = rng.normal(size=(1, h, d)), rng.normal(size=(1, d, h))
    b1, b2 = rng.normal(size=(1, h)), rng.normal(size=(1, d))
    Wg, Wn = rng.normal(size=(d, 1)), rng.normal(size=(d, 1))
    out = oracle.forward(x, Wg, Wn, None, rng.normal(size=(T, 1)), W1, b1, W2, b2, k=1)
    tx = torch.from_numpy(x)
    hid = torch.relu(torch.nn.functional.linear(tx, torch.from_numpy(W1[0]), torch.from_numpy(b1[0])))
    ref = torch.nn.functional.linear(hid, torch.from_numpy(W2[0]), torch.from_numpy(b2[0])).numpy()
    np.testing.assert_allclose(out["y"], ref, rtol=1e-12, atol=1e-12)
    assert np.all(out["G"] == 1.0) and np.all(out["idx"] == 0)
    for t in range(3):
        np.testing.assert_allclose(oracle.expert(x[t], W1[0], b1[0], W2[0], b2[0]), ref[t],
                                   rtol=1e-12, atol=1e-12)


def test_dense_mixture_when_k_equals_n():
    # k = n keeps every expert: y = sum_i softmax(H)_i E_i(x), the dense soft mixture.
    rng = np.random.default_rng(12)
    T, d, h, n = 10, 8, 12, 5
    x = rng.normal(size=(T, d))
    W1, W2 = rng.normal(size=(n, h, d)), rng.normal(size=(n, d, h))
    b1, b2 = rng.normal(size=(n, h)), rng.normal(size=(n, d))
    Wg, Wn = rng.normal(size=(d, n)), rng.normal(size=(d, n))
    out = oracle.forward(x, Wg, Wn, None, None, W1, b1, W2, b2, k=n)
    tx = torch.from_numpy(x)
    P = torch.softmax(tx @ torch.from_numpy(Wg), dim=1)
    ref = torch.zeros(T, d, dtype=torch.float64)
    for e in range(n):
        hid = torch.relu(torch.nn.functional.linear(tx, torch.from_numpy(W1[e]), torch.from_numpy(b1[e])))
        ref += P[:, e:e + 1] * torch.nn.functional.linear(hid, torch.from_numpy(W2[e]),
                                                          torch.from_numpy(b2[e]))
    np.testing.assert_allclose(out["y"], ref.numpy(), rtol=1e-11, atol=1e-11)
    Gd = np.zeros((T, n))
    np.put_along_axis(Gd, out["idx"], out["G"], axis=1)
    np.testing.assert_allclose(Gd, P.numpy(), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(out["importance"], P.numpy().sum(0), rtol=1e-12)


def test_combine_uses_only_selected_experts():
    # Poison an expert no token selects: y must not change.
    rng = np.random.default_rng(13)
    T, d, h, n, k = 12, 8, 8, 6, 2
    x = rng.normal(size=(T, d))
    W1, W2 = rng.normal(size=(n, h, d)), rng.normal(size=(n, d, h))
    b1, b2 = np.zeros((n, h)), np.zeros((n, d))
    Wg = rng.normal(size=(d, n))
    bg = np.zeros(n)
    bg[5] = -1e9                   # expert 5 is never among the top k
    out = oracle.forward(x, Wg, np.zeros_like(Wg), bg, None, W1, b1, W2, b2, k=k)
    assert out["counts"][5] == 0
    W1p = W1.copy()
    W1p[5] = np.nan
    out2 = oracle.forward(x, Wg, np.zeros_like(Wg), bg, None, W1p, b1, W2, b2, k=k)
    np.testing.assert_array_equal(out["y"], out2["y"])


def test_forward_hierarchical_invariants():
    rng = np.random.default_rng(14)
    T, d, h, G, m, kg, ki = 40, 8, 8, 4, 3, 2, 2
    n = G * m
    x = rng.normal(size=(T, d))
    Wg, Wn = rng.normal(size=(d, G + n)), rng.normal(size=(d, G + n))
    eps = rng.normal(size=(T, G + n))
    W1, W2 = rng.normal(size=(n, h, d)), rng.normal(size=(n, d, h))
    out = oracle.forward(x, Wg, Wn, None, eps, W1, np.zeros((n, h)), W2, np.zeros((n, d)),
                         k=kg * ki, groups=G, k_groups=kg)
    assert out["counts"].sum() == T * kg * ki
    assert out["importance"].sum() == pytest.approx(T, rel=1e-13)
    idx_h, G_h, _ = oracle.gate_hier(x, Wg, Wn, None, eps, G, kg, kg * ki)
    assert np.array_equal(out["idx"], idx_h)
    y = oracle.experts_combine(x, idx_h, G_h, W1, np.zeros((n, h)), W2, np.zeros((n, d)))
    np.testing.assert_array_equal(out["y"], y)


# --------------------------------------------------------------------------
# Combine from expert-order rows ("MoE:稀疏门控混合专家", section 二: y is the
# gate-weighted sum of the selected experts' outputs; only they contribute).
# --------------------------------------------------------------------------
def _combine_case(T=37, k=3, d=5, S_extra=4, drop=4, seed=3):
    """Expert-order rows Y [S, d], gate weights G [T, k] and an inv_perm that
    is a random permutation of the slots into rows, a few slots set to -1."""
    rng = np.random.default_rng(seed)
    S = T * k + S_extra
    Y = rng.normal(size=(S, d))
    G = rng.uniform(0.05, 1.0, size=(T, k))
    inv = rng.permutation(S)[: T * k].astype(np.int32)
    inv[rng.choice(T * k, size=drop, replace=False)] = -1
    return Y, G, inv


def _combine_pins(y, Y, G, inv):
    """Checks of a candidate combine result that do not restate its formula:
    (1) it equals the product of a scipy sparse [T, S] routing matrix with Y;
    (2) with Y the identity, row t holds G[t, j] at column inv[t*k+j];
    (3) with one-hot gate weights, row t is the selected expert row itself."""
    import scipy.sparse as sp
    T, k = G.shape
    S, d = Y.shape
    t_of = np.repeat(np.arange(T), k)
    keep = inv >= 0
    M = sp.csr_matrix((G.reshape(-1)[keep], (t_of[keep], inv[keep])), shape=(T, S))
    ok = np.allclose(y(Y, inv, G), M @ Y, rtol=1e-13, atol=1e-13)
    eye = np.eye(S)
    yi = y(eye, inv, G)
    want = np.zeros((T, S))
    for s in np.nonzero(keep)[0]:
        want[s // k, inv[s]] += G.reshape(-1)[s]
    ok &= np.array_equal(yi, want)
    for j in range(k):
        oh = np.zeros_like(G)
        oh[:, j] = 1.0
        rows = inv.reshape(T, k)[:, j]
        exp = np.where((rows >= 0)[:, None], Y[np.clip(rows, 0, None)], 0.0)
        ok &= np.array_equal(y(Y, inv, oh), exp)
    return bool(ok)


def test_combine_rows_pins():
    Y, G, inv = _combine_case()
    assert _combine_pins(oracle.combine_rows, Y, G, inv)


def test_combine_rows_pins_fail_planted_mistakes():
    # Plausible mistakes, planted in copies of the combine on the CPU: each
    # must fail the pins above.
    Y, G, inv = _combine_case(seed=5)

    def weight_dropped(Y_, inv_, G_):
        return oracle.combine_rows(Y_, inv_, np.ones_like(G_))

    def rows_by_slot(Y_, inv_, G_):
        T, k = G_.shape
        slot = np.where(inv_ >= 0, np.arange(T * k), -1).astype(np.int32)
        return oracle.combine_rows(Y_, slot, G_)

    def weight_of_next_slot(Y_, inv_, G_):
        return oracle.combine_rows(Y_, inv_, np.roll(G_, 1, axis=1))

    for bad in (weight_dropped, rows_by_slot, weight_of_next_slot):
        assert not _combine_pins(bad, Y, G, inv), bad.__name__


def test_combine_rows_composes_to_the_pinned_forward():
    # routing, the experts on expert-order rows and the combine give the same
    # y as the forward pass (itself pinned to torch's dense mixture and linear)
    rng = np.random.default_rng(9)
    T, d, h, n, k = 23, 16, 24, 5, 2
    x = rng.normal(size=(T, d))
    Wg = rng.normal(size=(d, n)) / math.sqrt(d)
    W1 = rng.normal(size=(n, h, d)) / math.sqrt(d)
    b1 = rng.normal(size=(n, h)) * 0.1
    W2 = rng.normal(size=(n, d, h)) / math.sqrt(h)
    b2 = rng.normal(size=(n, d)) * 0.1
    ref = oracle.forward(x, Wg, None, None, None, W1, b1, W2, b2, k)
    counts, offsets, perm, inv, imp, cv2 = oracle.route(ref["idx"], ref["G"], n)
    experts = ref["idx"].reshape(-1)[perm]
    Y = oracle.expert_rows(x[perm // k], experts, W1, b1, W2, b2)
    y = oracle.combine_rows(Y, inv, ref["G"])
    np.testing.assert_allclose(y, ref["y"], rtol=1e-12, atol=1e-12)


def test_combine_rows_rejects_a_row_out_of_range():
    Y, G, inv = _combine_case()
    bad = inv.copy()
    bad[7] = Y.shape[0]
    with pytest.raises(ValueError):
        oracle.combine_rows(Y, bad, G)
