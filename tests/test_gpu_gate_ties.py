"""Exact ties in the gate's KeepTopK ("MoE:稀疏门控混合专家", section 三:
keep the k largest scores; this library breaks equal scores by the lower
expert index, as the oracle does).

Columns of W_g are repeated so that whole groups of experts score exactly
the same for every token (identical columns give bit-identical products on
both sides); the tensor-core gate must then pick the same, lowest-index
members of each tied group as the oracle, through every stage of its
selection (first-chunk network, per-part insertion, the shared threshold
between parts, the merge of the parts).  Ties are exact on both sides;
scores that differ only near fp32 rounding are not, so tokens whose distinct
scores around the cut are closer than 1e-3 are left out of the comparison.
The all-zero gate makes every score equal: the choice is experts 0..k-1
with weights 1/k.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL_G, to_dev
from sparsely_gated_mixture_top_b300 import binding as B
from sparsely_gated_mixture_top_b300 import workloads as wl

pytestmark = pytest.mark.gpu


def run(w, Wg):
    inp = wl.make_inputs(w)
    inp["Wg"] = torch.from_numpy(Wg)
    d = to_dev(inp)
    s = B.shape_of(w)
    ws = B.workspace(s)
    idx = torch.empty((w.T, w.k), dtype=torch.int32, device="cuda")
    G = torch.empty((w.T, w.k), dtype=torch.float32, device="cuda")
    B.moe_gate(s, d["x"], d["Wg"], d["Wn"], d["bg"], d["eps"], idx, G, ws)
    assert B.moe_check(ws) == B.MOE_OK
    ref_idx, ref_G, H, _ = oracle.gate_flat(inp["x"], Wg, None, None, None, w.k)
    return idx.cpu().numpy(), G.cpu().double().numpy(), ref_idx, ref_G, H


def separated_rows(H, k, tol=1e-3):
    """Rows whose distinct scores, from the best down to the first one below
    the k-th, are at least tol apart (relative to max(1, |score|))."""
    keep = np.zeros(len(H), bool)
    for t, row in enumerate(H):
        s = np.sort(row)[::-1]
        u = np.unique(s)[::-1]
        pos = int(np.nonzero(u == s[k - 1])[0][0])
        cand = u[:pos + 2]
        keep[t] = bool(np.all(-np.diff(cand) >= tol * np.maximum(1.0, np.abs(cand[1:]))))
    return keep


@pytest.mark.parametrize("rep,k,n", [(2, 4, 256), (4, 4, 256), (8, 4, 512), (3, 2, 96),
                                     (16, 4, 256)])
def test_repeated_columns_pick_the_lowest_index(rep, k, n):
    w = wl.Workload("ties", T=700, d=512, h=256, n=n, k=k, noisy=False, seed=500 + rep)
    # unit-scale scores (the layer's own scale): columns ~ N(0, 1/d)
    base = (np.random.default_rng(rep).standard_normal((w.d, -(-n // rep))) /
            np.sqrt(w.d)).astype(np.float32)
    Wg = np.repeat(base, rep, axis=1)[:, :n].copy()
    idx, G, ref_idx, ref_G, H = run(w, Wg)
    keep = separated_rows(H, k)
    assert keep.mean() >= 0.8
    np.testing.assert_array_equal(idx[keep], ref_idx[keep])
    assert np.abs(G[keep] - ref_G[keep]).max() <= TOL_G


def test_all_scores_equal():
    w = wl.Workload("flat_zero", T=300, d=512, h=256, n=256, k=4, noisy=False, seed=7)
    idx, G, ref_idx, _, _ = run(w, np.zeros((w.d, w.n), np.float32))
    np.testing.assert_array_equal(idx, np.tile(np.arange(w.k), (w.T, 1)))
    np.testing.assert_array_equal(ref_idx, idx)
    np.testing.assert_allclose(G, 0.25, rtol=0, atol=1e-7)
