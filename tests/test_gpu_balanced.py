"""Parity of the layer with balanced routing (moe_forward_balanced, through
the C ABI) with the oracle ("Outrageously Large Neural Networks - 中文验证版",
section 方法适配: equal batch sizes per expert in training by a per-batch mask,
per-expert thresholds at inference).

The mask is index work and must match the oracle's exactly.  The CUDA scores
are fp32 and the oracle's fp64, so the inputs are made to have one right
answer: every column's cut (between the kept and the first dropped score)
has a gap of at least 1e-3 in the oracle's scores, single eps cells being
redrawn until it does (noise-off cases use a seed whose gaps already clear
it).  Thresholds are placed by the oracle's scores midway across such a gap,
never taken from the CUDA side.  Then: masks and counts identical, weights
within 1e-5, y within the forward's bars (2e-2 relative Frobenius in bf16,
1e-4 in fp32).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.margin import column_cut_gaps, enforce_cut_margin
from parity_util import TOL_Y, rel_fro, to_dev
from sparsely_gated_mixture_top_b300 import binding as B
from sparsely_gated_mixture_top_b300 import workloads as wl

pytestmark = pytest.mark.gpu

W = wl.Workload
CASES = [
    (W("bal_bf16_batchwise", T=600, d=256, h=512, n=12, k=2, bias_std=0.1, seed=61), None),
    (W("bal_f32_batchwise", T=300, d=128, h=128, n=8, k=3, dtype="f32", bias_std=0.1, seed=62), None),
    (W("bal_noise_off", T=400, d=128, h=256, n=6, k=2, noisy=False, seed=63), None),
    (W("bal_zipf_batchwise", T=2000, d=128, h=128, n=16, k=2, gate_bias="zipf", seed=64), None),
    (W("bal_ragged_m", T=333, d=64, h=128, n=7, k=2, seed=65), None),   # k*T/n not whole
    (W("bal_bf16_thresholds", T=600, d=256, h=512, n=12, k=2, bias_std=0.1, seed=66), "quantile"),
    (W("bal_f32_thresholds", T=300, d=128, h=128, n=8, k=3, dtype="f32", seed=67), "quantile"),
]


@pytest.fixture(autouse=True)
def _free_cuda():
    yield
    torch.cuda.empty_cache()


def cut_between(col, rank):
    """A threshold midway between the rank-th and (rank+1)-th largest of col."""
    s = np.sort(col)[::-1]
    return 0.5 * (s[rank - 1] + s[rank]) if 0 < rank < len(s) else (s[0] + 1.0 if rank == 0 else s[-1] - 1.0)


def run(w, dinp, thr, rows_cap):
    s = B.shape_of(w)
    ws = B.balanced_workspace(s, rows_cap)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    y = torch.full((w.T, w.d), float("nan"), dtype=dt, device="cuda")
    counts = torch.full((w.n,), -1, dtype=torch.int32, device="cuda")
    Wd = torch.full((w.T, w.n), float("nan"), device="cuda")
    thr_d = torch.from_numpy(thr.astype(np.float32)).cuda() if thr is not None else None
    B.moe_forward_balanced(s, dinp["x"], dinp["Wg"], dinp["Wn"], dinp["bg"],
                           dinp["eps"] if w.noisy else None, thr_d, rows_cap, dinp["W1"],
                           dinp["b1"], dinp["W2"], dinp["b2"], y, counts, Wd, ws)
    status = B.moe_check(ws)
    assert status == B.MOE_OK, B.status_string(status)
    return y.cpu().double().numpy(), counts.cpu().numpy(), Wd.cpu().double().numpy()


def compare(got, ref, tol_y):
    y, counts, Wg_ = got
    keep_g, keep_r = Wg_ > 0, ref["W"] > 0
    np.testing.assert_array_equal(keep_g, keep_r)
    np.testing.assert_array_equal(counts, keep_r.sum(axis=0))
    np.testing.assert_allclose(Wg_, ref["W"], atol=1e-5, rtol=0)
    assert rel_fro(y, ref["y"]) <= tol_y
    return keep_g


def clear_cuts(w, inp, ranks, margin=1e-3):
    """Make every column's cut at its rank unambiguous (see the module notes)."""
    if w.noisy:
        enforce_cut_margin(w, inp, ranks, margin)
    _, _, H, _ = oracle.gate_flat(inp["x"], inp["Wg"], inp["Wn"], inp["bg"],
                                  inp["eps"] if w.noisy else None, 1)
    assert column_cut_gaps(H, ranks).min() >= margin
    return H


@pytest.mark.parametrize("w,mode", CASES, ids=[c[0].name for c in CASES])
def test_balanced_matches_oracle(w, mode):
    inp = wl.make_inputs(w)
    m = w.k * w.T // w.n
    if mode is None:
        ranks = [m] * w.n
    else:
        # per-expert cuts at different quantiles, so the counts differ
        ranks = [max(1, (e + 1) * w.T // (w.n + 2)) for e in range(w.n)]
    H = clear_cuts(w, inp, ranks)
    dinp = to_dev(inp)
    if mode is None:
        thr = None
        rows_cap = w.n * m
    else:
        thr = np.array([cut_between(H[:, e], r) for e, r in enumerate(ranks)])
        rows_cap = int(sum(ranks)) + 7
    ref = oracle.forward_balanced(inp["x"], inp["Wg"], inp["Wn"], inp["bg"],
                                  inp["eps"] if w.noisy else None, thr, inp["W1"], inp["b1"],
                                  inp["W2"], inp["b2"], w.k)
    got = run(w, dinp, thr, rows_cap)
    keep = compare(got, ref, TOL_Y[w.dtype])
    np.testing.assert_array_equal(keep.sum(axis=0), ranks)
    # weights of every token sum to 1 over its kept experts (0 when none)
    sums = got[2].sum(axis=1)
    kept_any = keep.any(axis=1)
    assert np.all(np.abs(sums[kept_any] - 1.0) <= 1e-5) and not sums[~kept_any].any()


def test_threshold_overflow_is_reported():
    w = W("bal_overflow", T=200, d=64, h=64, n=4, k=2, seed=68)
    dinp = to_dev(wl.make_inputs(w))
    s = B.shape_of(w)
    cap = 50
    ws = B.balanced_workspace(s, cap)
    y = torch.empty((w.T, w.d), dtype=torch.bfloat16, device="cuda")
    counts = torch.empty((w.n,), dtype=torch.int32, device="cuda")
    thr = torch.full((w.n,), -1e30, device="cuda")       # every expert keeps every token
    B.moe_forward_balanced(s, dinp["x"], dinp["Wg"], dinp["Wn"], dinp["bg"], dinp["eps"], thr, cap,
                           dinp["W1"], dinp["b1"], dinp["W2"], dinp["b2"], y, counts, None, ws)
    assert B.moe_check(ws) == B.MOE_ERR_DEVICE
    assert (counts.cpu().numpy() == w.T).all()


def test_full_size_batchwise():
    """flat_n256_k4 (T=16384, n=256, k=4): every expert keeps m = 256 tokens;
    the whole mask against the oracle's scores, exactly; y of 64 sampled
    tokens against the oracle run on those tokens alone with each expert's cut
    placed between its m-th and (m+1)-th score of the whole batch (the same
    mask)."""
    w = wl.WORKLOADS["flat_n256_k4"]
    inp = wl.make_inputs(w)
    m = w.k * w.T // w.n
    H = clear_cuts(w, inp, [m] * w.n)
    dinp = to_dev(inp)
    y, counts, Wd = run(w, dinp, None, w.n * m)
    assert (counts == m).all()
    srt = -np.sort(-H, axis=0)
    keep_r = H >= srt[m - 1][None, :]
    np.testing.assert_array_equal(Wd > 0, keep_r)
    rng = np.random.default_rng(9)
    tokens = np.sort(rng.choice(w.T, 64, replace=False))
    thr = 0.5 * (srt[m - 1] + srt[m])
    sub = {k: (v[tokens] if k in ("x", "eps") and v is not None else v) for k, v in inp.items()}
    ref = oracle.forward_balanced(sub["x"], sub["Wg"], sub["Wn"], sub["bg"], sub["eps"], thr,
                                  sub["W1"], sub["b1"], sub["W2"], sub["b2"], w.k)
    np.testing.assert_array_equal(Wd[tokens] > 0, ref["W"] > 0)
    np.testing.assert_allclose(Wd[tokens], ref["W"], atol=1e-5, rtol=0)
    assert rel_fro(y[tokens], ref["y"]) <= TOL_Y[w.dtype]
