"""Parity of the backward pass (moe_backward, through the C ABI) with the CPU
oracle's backward (fp64, pinned by finite differences of the oracle forward).

The CUDA backward takes the selection (idx, G, importance) of the CUDA
forward; the oracle runs its own gate, and the two selections are checked to
be identical first.  Shapes that run on the CUDA cores compute every gradient
in fp32 from the exact stored inputs: the bar is a relative Frobenius error of
1e-4 (fp32 rounding over sums of at most a few thousand terms, against fp64).
bf16 shapes with widths that are multiples of 128 run the contractions on the
tensor cores with bf16 operands and bf16 intermediates (E, dE, dZ, dX rows),
the precision of the forward's expert stage: the bar is the forward's bf16
bar, 2e-2.  Small cases compare every element; the full-size
default workload compares the gradients of three whole experts and of a
sample of tokens (without the importance term, each of those depends only on
the tokens that chose the expert, or on the token itself, so the oracle
computes them on that subset alone) and checks properties of the rest.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import prepared_inputs, rel_fro, run_forward, to_dev
from sparsely_gated_mixture_top_b300 import binding as B
from sparsely_gated_mixture_top_b300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = 1e-4
TOL_TC = 2e-2
GRADS = ("dx", "dWg", "dWn", "dbg", "dW1", "db1", "dW2", "db2")

W = wl.Workload
CASES = [
    (W("bwd_bf16_ragged", T=37, d=64, h=128, n=5, k=2, bias_std=0.1, seed=41), 0.7),
    (W("bwd_f32_ragged", T=37, d=64, h=128, n=5, k=2, dtype="f32", bias_std=0.1, seed=42), 0.7),
    (W("bwd_bf16_tiles", T=600, d=192, h=320, n=7, k=3, bias_std=0.05, seed=43), 1.5),
    (W("bwd_k1", T=100, d=64, h=64, n=6, k=1, bias_std=0.1, seed=44), 0.3),
    (W("bwd_dense_k_eq_n_f32", T=64, d=128, h=128, n=8, k=8, dtype="f32", seed=45), 2.0),
    (W("bwd_noise_off", T=80, d=64, h=128, n=6, k=2, noisy=False, seed=46), 0.5),
    (W("bwd_many_empty_experts", T=20, d=128, h=256, n=64, k=2, seed=47), 1.0),
    (W("bwd_zipf_empty_experts", T=2500, d=256, h=256, n=200, k=4, gate_bias="zipf", seed=48), 0.2),
    (W("bwd_no_aux_loss_k16", T=50, d=64, h=64, n=20, k=16, seed=49), 0.0),
    # tensor-core path (bf16, widths multiples of 128)
    (W("bwd_tc_ragged", T=600, d=256, h=512, n=7, k=3, bias_std=0.05, seed=51), 1.5),
    (W("bwd_tc_k1", T=300, d=128, h=128, n=6, k=1, bias_std=0.1, seed=52), 0.3),
    (W("bwd_tc_noise_off", T=300, d=128, h=256, n=6, k=2, noisy=False, seed=53), 0.5),
    (W("bwd_tc_k16", T=200, d=128, h=128, n=20, k=16, seed=54), 0.0),
    (W("bwd_tc_wide_experts", T=700, d=512, h=1024, n=3, k=1, bias_std=0.1, seed=55), 0.4),
    (W("bwd_tc_k8", T=200, d=256, h=256, n=20, k=8, bias_std=0.1, seed=56), 0.6),
    # hierarchical gate (the 16 x 256 scheme of "MoE:稀疏门控混合专家", section 三,
    # at test sizes): both softmax levels, group and expert columns
    (W("bwd_hier_f32", T=120, d=64, h=128, n=16, k=4, groups=4, k_groups=2, dtype="f32",
       bias_std=0.1, seed=61), 0.8),
    (W("bwd_hier_bf16_cuda_cores", T=150, d=64, h=128, n=24, k=4, groups=6, k_groups=2,
       seed=62), 0.5),
    (W("bwd_hier_tc", T=400, d=256, h=512, n=64, k=4, groups=8, k_groups=2, bias_std=0.05,
       seed=63), 1.0),
    (W("bwd_hier_tc_one_group_kept", T=300, d=128, h=256, n=32, k=4, groups=4, k_groups=1,
       seed=64), 0.3),
    (W("bwd_hier_one_expert_per_group", T=100, d=128, h=128, n=16, k=2, groups=8, k_groups=2,
       seed=65), 0.4),
    (W("bwd_hier_k8_f32", T=100, d=64, h=64, n=32, k=8, groups=4, k_groups=2, dtype="f32",
       seed=66), 0.6),
]


def tol(w):
    tc = w.dtype == "bf16" and w.d % 128 == 0 and w.h % 128 == 0
    return TOL_TC if tc else TOL


@pytest.fixture(autouse=True)
def _free_cuda():
    yield
    torch.cuda.empty_cache()


def make_dy(w, T=None, seed=None):
    T = w.T if T is None else T
    rng = np.random.default_rng(1000 + (w.seed if seed is None else seed))
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    return torch.from_numpy(rng.normal(size=(T, w.d)).astype(np.float32)).to(dt)


def run_backward(w, dinp, fwd, dy, w_imp):
    s = B.shape_of(w)
    ws = B.backward_workspace(s)
    T, d, h, n = w.T, w.d, w.h, w.n
    C = n + w.groups   # gate score columns, the group columns first

    def f32(*shape):
        return torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")

    g = dict(dx=f32(T, d), dWg=f32(d, C), dWn=f32(d, C), dbg=f32(C), dW1=f32(n, h, d),
             db1=f32(n, h), dW2=f32(n, d, h), db2=f32(n, d))
    B.moe_backward(s, dinp["x"], dinp["Wg"], dinp["Wn"], dinp["eps"] if w.noisy else None,
                   dinp["W1"], dinp["b1"], dinp["W2"], dinp["b2"], fwd["idx"], fwd["G"],
                   fwd["importance"], dy.cuda(), w_imp, g["dx"], g["dWg"], g["dWn"], g["dbg"],
                   g["dW1"], g["db1"], g["dW2"], g["db2"], ws)
    status = B.moe_check(ws)
    assert status == B.MOE_OK, B.status_string(status)
    return {k: v.cpu().numpy() for k, v in g.items()}


def oracle_backward(w, inp, dy, w_imp):
    if w.groups:
        return oracle.backward_hier(inp["x"], inp["Wg"], inp["Wn"], inp["bg"],
                                    inp["eps"] if w.noisy else None, inp["W1"], inp["b1"],
                                    inp["W2"], inp["b2"], dy, w.k, w.groups, w.k_groups, w_imp)
    return oracle.backward(inp["x"], inp["Wg"], inp["Wn"], inp["bg"],
                           inp["eps"] if w.noisy else None, inp["W1"], inp["b1"], inp["W2"],
                           inp["b2"], dy, w.k, w_imp)


@pytest.mark.parametrize("w,w_imp", CASES, ids=[c[0].name for c in CASES])
def test_backward_matches_oracle(w, w_imp):
    inp = prepared_inputs(w)
    dinp = to_dev(inp)
    fwd, _ = run_forward(w, dinp)
    dy = make_dy(w)
    got = run_backward(w, dinp, fwd, dy, w_imp)
    ref = oracle_backward(w, inp, dy, w_imp)
    np.testing.assert_array_equal(fwd["idx"].cpu().numpy(), ref["idx"])
    for key in GRADS:
        assert np.isfinite(got[key]).all(), key
        err = rel_fro(got[key], ref[key])
        assert err <= tol(w), (key, err)
    if not w.noisy:
        assert not got["dWn"].any()
    if w.k == 1:
        assert not got["dWg"].any() and not got["dbg"].any()
    if w.groups:
        # both softmaxes are shift invariant: the bias gradients of the group
        # columns sum to zero, and so do those of each group's own columns
        m, G = w.n // w.groups, w.groups
        scale = 1.0 + np.abs(got["dbg"]).sum()
        assert abs(float(got["dbg"][:G].sum())) <= 1e-4 * scale
        for grp in range(G):
            assert abs(float(got["dbg"][G + grp * m:G + (grp + 1) * m].sum())) <= 1e-4 * scale


@pytest.mark.parametrize("case", [2, 9], ids=["cuda_cores", "tensor_cores"])
def test_backward_is_deterministic(case):
    w, w_imp = CASES[case]
    inp = prepared_inputs(w)
    dinp = to_dev(inp)
    fwd, _ = run_forward(w, dinp)
    dy = make_dy(w)
    a = run_backward(w, dinp, fwd, dy, w_imp)
    b = run_backward(w, dinp, fwd, dy, w_imp)
    for key in GRADS:
        np.testing.assert_array_equal(a[key], b[key])


def test_backward_of_empty_input_is_zero():
    w = W("bwd_empty", T=0, d=64, h=64, n=4, k=2, seed=50)
    s = B.shape_of(w)
    ws = B.backward_workspace(s)
    dev = "cuda"
    nan = lambda *sh: torch.full(sh, float("nan"), device=dev)  # noqa: E731
    Wg, Wn = torch.zeros(64, 4, device=dev), torch.zeros(64, 4, device=dev)
    W1 = torch.zeros(4, 64, 64, dtype=torch.bfloat16, device=dev)
    W2 = torch.zeros(4, 64, 64, dtype=torch.bfloat16, device=dev)
    g = dict(dWg=nan(64, 4), dWn=nan(64, 4), dbg=nan(4), dW1=nan(4, 64, 64), db1=nan(4, 64),
             dW2=nan(4, 64, 64), db2=nan(4, 64))
    B.moe_backward(s, None, Wg, Wn, None, W1, None, W2, None, None, None, None, None, 0.0, None,
                   g["dWg"], g["dWn"], g["dbg"], g["dW1"], g["db1"], g["dW2"], g["db2"], ws)
    assert B.moe_check(ws) == B.MOE_OK
    for key, v in g.items():
        assert not v.any(), key


def test_full_size_workload_sampled():
    """flat_n256_k4 (T=16384, d=512, h=1024, n=256, k=4), no importance term:
    three whole experts (fewest, median and most rows) and 64 tokens against
    the oracle on their own token subsets; properties of all gradients."""
    w = wl.WORKLOADS["flat_n256_k4"]
    inp = prepared_inputs(w)
    dinp = to_dev(inp)
    fwd, _ = run_forward(w, dinp)
    dy = make_dy(w)
    got = run_backward(w, dinp, fwd, dy, 0.0)
    for key in GRADS:
        assert np.isfinite(got[key]).all(), key
    # the oracle's own selection decides which tokens each expert saw
    idx_ref, _, _, _ = oracle.gate_flat(inp["x"], inp["Wg"], inp["Wn"], inp["bg"], inp["eps"], w.k)
    np.testing.assert_array_equal(fwd["idx"].cpu().numpy(), idx_ref)
    counts = np.bincount(idx_ref.ravel(), minlength=w.n)
    order = np.argsort(counts, kind="stable")
    experts = [int(order[0]), int(order[w.n // 2]), int(order[-1])]

    def sub(rows):
        return {k: (v[rows] if k in ("x", "eps") and v is not None else v) for k, v in inp.items()}

    for e in experts:
        rows = np.nonzero((idx_ref == e).any(axis=1))[0]
        ref = oracle_backward(w, sub(rows), dy[torch.from_numpy(rows)], 0.0)
        for key in ("dW1", "db1", "dW2", "db2"):
            assert rel_fro(got[key][e], ref[key][e]) <= tol(w), (e, key)
        for key in ("dWg", "dWn"):
            assert rel_fro(got[key][:, e], ref[key][:, e]) <= tol(w), (e, key)
        assert abs(got["dbg"][e] - ref["dbg"][e]) <= tol(w) * (1 + abs(ref["dbg"][e]))
    rng = np.random.default_rng(7)
    tokens = np.sort(rng.choice(w.T, 64, replace=False))
    ref = oracle_backward(w, sub(tokens), dy[torch.from_numpy(tokens)], 0.0)
    assert rel_fro(got["dx"][tokens], ref["dx"]) <= tol(w)
    # softmax shift invariance: the gate bias gradients sum to zero
    assert abs(float(got["dbg"].astype(np.float64).sum())) <= 1e-3 * float(np.abs(got["dbg"]).sum())
