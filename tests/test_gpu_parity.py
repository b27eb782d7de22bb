"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Small cases compare every output of every token; they span several tiles,
ragged tails, experts with no rows, one expert taking every token, the dense
k = n mixture, a single expert, empty input, both dtypes and both gating
variants.  The full-size workloads compare sampled tokens with the oracle
and check the routing outputs of all tokens by properties that hold at any
size.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import (TOL_G, TOL_Y, check_against_oracle, check_routing_properties,
                         gate_margins, oracle_full, prepared_inputs, rel_fro, run_components,
                         run_forward, sampled_oracle, to_dev)
from sparsely_gated_mixture_top_b300 import binding as B
from sparsely_gated_mixture_top_b300 import workloads as wl

pytestmark = pytest.mark.gpu

W = wl.Workload
SMALL = [
    W("flat_bf16_ragged", T=37, d=64, h=128, n=5, k=2, bias_std=0.1, seed=11),
    W("flat_f32_ragged", T=37, d=64, h=128, n=5, k=2, dtype="f32", bias_std=0.1, seed=12),
    W("flat_bf16_tiles", T=1000, d=192, h=320, n=7, k=3, bias_std=0.05, seed=13),
    W("flat_f32_tiles", T=300, d=192, h=320, n=7, k=3, dtype="f32", seed=14),
    W("single_token_single_expert", T=1, d=64, h=64, n=1, k=1, seed=15),
    W("dense_k_eq_n_bf16", T=200, d=128, h=256, n=8, k=8, seed=16),
    W("dense_k_eq_n_f32", T=64, d=128, h=256, n=8, k=8, dtype="f32", seed=17),
    W("many_empty_experts", T=20, d=128, h=256, n=64, k=2, seed=18),
    W("hier_bf16", T=300, d=128, h=256, n=32, k=4, groups=4, k_groups=2, bias_std=0.1, seed=19),
    W("hier_f32", T=100, d=128, h=256, n=32, k=4, groups=4, k_groups=2, dtype="f32", seed=20),
    W("hier_one_group", T=64, d=64, h=128, n=12, k=3, groups=1, k_groups=1, seed=21),
    W("wide_k16", T=128, d=64, h=128, n=40, k=16, seed=22),
    W("bn256_two_tiles", T=700, d=512, h=1024, n=3, k=1, bias_std=0.1, seed=23),
    W("hier_wide_inner_cuda_core_gate", T=50, d=64, h=64, n=32, k=8, groups=2, k_groups=1,
      seed=24),
    W("hier_stream_x", T=130, d=576, h=128, n=12, k=2, groups=3, k_groups=1, seed=25),
    W("flat_stream_x_k1", T=300, d=640, h=64, n=70, k=1, bias_std=0.1, seed=26),
    W("big_experts_ragged", T=1500, d=256, h=512, n=5, k=2, bias_std=0.3, seed=27),
    W("zipf_sparse_tail", T=4000, d=256, h=256, n=16, k=1, gate_bias="zipf", seed=28),
    # Thousands of slots: many 128-row blocks per expert with ragged and
    # exactly full last blocks, 96 experts with no rows beside one with 2424,
    # and the FFN widths of the full-size workloads.
    W("many_blocks_ragged", T=3000, d=256, h=512, n=24, k=4, bias_std=0.2, seed=29),
    W("zipf_empty_experts", T=2500, d=256, h=256, n=200, k=4, gate_bias="zipf", seed=30),
    W("full_widths_16_experts", T=2400, d=512, h=1024, n=16, k=4, bias_std=0.1, seed=31),
    # Both expert layers in one kernel (at most 128 rows per expert on
    # average): one hidden chunk and two output blocks; an odd number of
    # hidden chunks with experts of a few rows (tiles of 32 columns, 16 token
    # rows per SM of the pair); the full widths with experts of one to three
    # token tiles.
    W("fused_one_chunk", T=600, d=512, h=256, n=12, k=2, bias_std=0.1, seed=32),
    W("fused_short_tiles_odd_chunks", T=40, d=256, h=768, n=24, k=3, bias_std=0.1, seed=33),
    W("fused_full_widths", T=2000, d=512, h=1024, n=64, k=4, bias_std=0.1, seed=34),
]


@pytest.fixture(autouse=True)
def _free_cuda():
    yield
    torch.cuda.empty_cache()


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_forward_matches_oracle_small(w):
    inp = prepared_inputs(w)
    ref = oracle_full(w, inp)
    out, ws = run_forward(w, to_dev(inp))
    check_against_oracle(w, out, ref)


@pytest.mark.parametrize("w", [SMALL[0], SMALL[1], SMALL[2], SMALL[8]],
                         ids=lambda w: w.name)
def test_components_match_oracle_and_forward(w):
    inp = prepared_inputs(w)
    ref = oracle_full(w, inp)
    dinp = to_dev(inp)
    r = run_components(w, dinp)
    np.testing.assert_array_equal(r["idx"].cpu().numpy(), ref["idx"])
    assert np.abs(r["G"].cpu().double().numpy() - ref["G"]).max() <= TOL_G
    np.testing.assert_array_equal(r["counts"].cpu().numpy(), ref["counts"])
    np.testing.assert_array_equal(r["offsets"].cpu().numpy(), ref["offsets"])
    np.testing.assert_array_equal(r["perm"].cpu().numpy(), ref["perm"])
    np.testing.assert_array_equal(r["inv_perm"].cpu().numpy(), ref["inv_perm"])
    # expert outputs row by row against the oracle's experts
    perm = ref["perm"]
    toks = perm // w.k
    ex = ref["idx"].reshape(-1)[perm]
    Yref = oracle.expert_rows(oracle._f64(inp["x"])[toks], ex, inp["W1"], inp["b1"], inp["W2"],
                              inp["b2"])
    assert rel_fro(r["Y"].cpu().double().numpy(), Yref) <= TOL_Y[w.dtype]
    assert rel_fro(r["y"].cpu().double().numpy(), ref["y"]) <= TOL_Y[w.dtype]
    # the fused call gives the same bits as the four component calls
    out, _ = run_forward(w, dinp)
    assert torch.equal(out["y"], r["y"]) and torch.equal(out["idx"], r["idx"])
    assert torch.equal(out["G"], r["G"]) and torch.equal(out["importance"], r["importance"])


def test_each_stage_on_oracle_inputs():
    """Every stage fed with oracle (not GPU) intermediates."""
    w = W("stages", T=250, d=128, h=192, n=9, k=3, bias_std=0.1, seed=31)
    inp = prepared_inputs(w)
    ref = oracle_full(w, inp)
    s = B.shape_of(w)
    ws = B.workspace(s)
    dinp = to_dev(inp)
    S = w.T * w.k
    idx = torch.from_numpy(ref["idx"]).cuda()
    G = torch.from_numpy(ref["G"]).float().cuda()
    counts = torch.empty(w.n, dtype=torch.int32, device="cuda")
    offsets = torch.empty(w.n + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(S, dtype=torch.int32, device="cuda")
    inv = torch.empty(S, dtype=torch.int32, device="cuda")
    imp = torch.empty(w.n, dtype=torch.float32, device="cuda")
    cv2 = torch.empty(1, dtype=torch.float32, device="cuda")
    B.moe_dispatch(s, idx, G, counts, offsets, perm, inv, imp, cv2, ws)
    np.testing.assert_array_equal(perm.cpu().numpy(), ref["perm"])
    np.testing.assert_array_equal(inv.cpu().numpy(), ref["inv_perm"])
    np.testing.assert_allclose(imp.cpu().double().numpy(), ref["importance"], rtol=1e-5)
    assert abs(cv2.item() - ref["cv2"]) <= 1e-4 * ref["cv2"]
    # FFN on the oracle's permutation
    Y = torch.empty((S, w.d), dtype=torch.bfloat16, device="cuda")
    rperm = torch.from_numpy(ref["perm"]).cuda()
    roff = torch.from_numpy(ref["offsets"]).cuda()
    B.moe_expert_ffn(s, dinp["x"], rperm, roff, dinp["W1"], dinp["b1"], dinp["W2"], dinp["b2"], Y, ws)
    toks = ref["perm"] // w.k
    ex = ref["idx"].reshape(-1)[ref["perm"]]
    Yref = oracle.expert_rows(oracle._f64(inp["x"])[toks], ex, inp["W1"], inp["b1"], inp["W2"],
                              inp["b2"])
    assert rel_fro(Y.cpu().double().numpy(), Yref) <= TOL_Y["bf16"]
    # combine on oracle expert rows (rounded to bf16 as the stage's input type)
    Yin = torch.from_numpy(Yref).to(torch.bfloat16).cuda()
    y = torch.empty((w.T, w.d), dtype=torch.bfloat16, device="cuda")
    rinv = torch.from_numpy(ref["inv_perm"]).cuda()
    B.moe_combine(s, Yin, rinv, G, y, ws)
    yref = oracle.combine_rows(Yin.cpu(), ref["inv_perm"].reshape(w.T, w.k), G.cpu())
    assert rel_fro(y.cpu().double().numpy(), yref) <= 1e-2 * 0.5
    assert B.moe_check(ws) == B.MOE_OK


def test_one_expert_takes_every_token():
    w = W("hot_expert", T=1000, d=128, h=256, n=4, k=2, seed=32)
    bg = torch.tensor([50.0, 0.0, 0.0, 0.0])
    inp = prepared_inputs(w, bg=bg)
    ref = oracle_full(w, inp)
    assert ref["counts"][0] == w.T
    out, _ = run_forward(w, to_dev(inp))
    check_against_oracle(w, out, ref)


def test_one_expert_takes_every_token_fused_ffn():
    """Both expert layers in one kernel (experts average at most 128 rows)
    while one expert holds all 1000 rows: eight token tiles of one expert."""
    w = W("hot_expert_fused", T=1000, d=256, h=512, n=8, k=1, bias_std=0.1, seed=36)
    bg = torch.tensor([50.0] + [0.0] * 7)
    inp = prepared_inputs(w, bg=bg)
    ref = oracle_full(w, inp)
    assert ref["counts"][0] == w.T
    out, _ = run_forward(w, to_dev(inp))
    check_against_oracle(w, out, ref)


@pytest.mark.parametrize("counts", [
    [128, 129, 0, 256, 1, 31, 32, 33],        # tiles: 128 | 80 + 49 | 2 x 128 | 1 row (N = 32)
    [0, 0, 0, 610, 0, 0, 0, 0],               # one expert: 4 x 128 + 98 rows
    [17, 15, 16, 14, 18, 13, 19, 498],        # tiles of 32 columns beside 3 x 128 + 114
], ids=["tile_edges", "one_expert", "small_tiles"])
def test_expert_stage_tile_edges_fused_ffn(counts):
    """moe_expert_ffn (the fused two-layer kernel at these widths) on chosen
    expert row counts and a shuffled slot order, against the oracle's
    experts applied to the same rows."""
    w = W("tile_edges", T=610, d=256, h=768, n=8, k=1, bias_std=0.1, seed=37)
    assert sum(counts) == w.T * w.k
    inp = wl.make_inputs(w)
    s = B.shape_of(w)
    ws = B.workspace(s)
    dinp = to_dev(inp)
    rng = np.random.default_rng(37)
    perm = rng.permutation(w.T * w.k).astype(np.int32)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    experts = np.repeat(np.arange(w.n), counts)
    Y = torch.empty((w.T * w.k, w.d), dtype=torch.bfloat16, device="cuda")
    B.moe_expert_ffn(s, dinp["x"], torch.from_numpy(perm).cuda(), torch.from_numpy(offsets).cuda(),
                     dinp["W1"], dinp["b1"], dinp["W2"], dinp["b2"], Y, ws)
    assert B.moe_check(ws) == B.MOE_OK
    Yref = oracle.expert_rows(oracle._f64(inp["x"])[perm // w.k], experts, inp["W1"], inp["b1"],
                              inp["W2"], inp["b2"])
    assert rel_fro(Y.cpu().double().numpy(), Yref) <= TOL_Y["bf16"]
    # every row individually (a row written to the wrong place fails here)
    err = np.abs(Y.cpu().double().numpy() - Yref).max(axis=1)
    scale = np.abs(Yref).max(axis=1) + 1e-3
    assert (err / scale).max() < 5e-2


def test_noise_off():
    w = W("clean_gate", T=500, d=128, h=192, n=16, k=2, noisy=False, seed=33)
    inp = wl.make_inputs(w)
    ref = oracle_full(w, inp)
    out, _ = run_forward(w, to_dev(inp))
    unique = gate_margins(w, inp, np.arange(w.T)) >= 1e-3
    assert unique.mean() > 0.95
    check_against_oracle(w, out, ref, tokens=unique)


def test_empty_input():
    w = W("empty", T=0, d=64, h=64, n=4, k=2, seed=34)
    s = B.shape_of(w)
    inp = to_dev(wl.make_inputs(w))
    ws = B.workspace(s)
    out = B.outputs(s)
    out["counts"].fill_(7)
    out["importance"].fill_(7)
    B.forward(s, inp, ws=ws, out=out)
    assert B.moe_check(ws) == B.MOE_OK
    assert out["counts"].sum().item() == 0 and out["importance"].abs().sum().item() == 0.0
    assert out["cv2"].item() == 0.0


def test_deterministic_bits():
    w = W("repeat", T=2000, d=256, h=512, n=32, k=4, seed=35)
    dinp = to_dev(prepared_inputs(w))
    a, _ = run_forward(w, dinp)
    b, _ = run_forward(w, dinp)
    for key in ("y", "G", "idx", "importance", "cv2", "counts"):
        assert torch.equal(a[key], b[key]), key


def test_out_of_range_expert_index_is_reported():
    w = W("bad_idx", T=64, d=64, h=64, n=8, k=2, seed=36)
    s = B.shape_of(w)
    ws = B.workspace(s)
    idx = torch.randint(0, 8, (64, 2), dtype=torch.int32, device="cuda")
    idx[5, 1] = 8
    idx[9, 0] = -3
    G = torch.full((64, 2), 0.5, device="cuda")
    S = 128
    counts = torch.empty(8, dtype=torch.int32, device="cuda")
    offsets = torch.empty(9, dtype=torch.int32, device="cuda")
    perm = torch.empty(S, dtype=torch.int32, device="cuda")
    inv = torch.empty(S, dtype=torch.int32, device="cuda")
    imp = torch.empty(8, device="cuda")
    cv2 = torch.empty(1, device="cuda")
    B.moe_dispatch(s, idx, G, counts, offsets, perm, inv, imp, cv2, ws)
    assert B.moe_check(ws) == B.MOE_ERR_DEVICE
    assert B.moe_check(ws) == B.MOE_OK          # cleared by the first read
    assert counts.sum().item() == S - 2
    assert inv[5 * 2 + 1].item() == -1 and inv[9 * 2].item() == -1
    valid = idx.reshape(-1).cpu().numpy()
    keep = (valid >= 0) & (valid < 8)
    p = perm.cpu().numpy()[:S - 2]
    np.testing.assert_array_equal(p, np.nonzero(keep)[0][np.argsort(valid[keep], kind="stable")])
    assert (perm.cpu().numpy()[S - 2:] == -1).all()


# --------------------------------------------------------------------------
# Full-size workloads, in the launch configuration the benchmark times.
# --------------------------------------------------------------------------
FULL = list(wl.WORKLOADS.values())


@pytest.mark.parametrize("w", FULL, ids=[w.name for w in FULL])
def test_full_size_workload(w):
    rng = np.random.default_rng(w.seed)
    full_oracle = w.T * w.k * w.d * w.h <= 16384 * 4 * 512 * 1024
    if full_oracle:
        rows = None
    else:
        nsamp = 256 if w.n >= 1024 else 384
        rows = np.unique(np.concatenate([[0, w.T - 1], rng.choice(w.T, nsamp, replace=False)]))
    inp = prepared_inputs(w, rows=rows)
    dinp = to_dev(inp)
    out, ws = run_forward(w, dinp)
    if full_oracle:
        ref = oracle_full(w, inp)
        check_against_oracle(w, out, ref)
    else:
        ref = sampled_oracle(w, inp, rows)
        idx = out["idx"].cpu().numpy()[rows]
        np.testing.assert_array_equal(idx, ref["idx"])
        assert np.abs(out["G"].cpu().double().numpy()[rows] - ref["G"]).max() <= TOL_G
        assert rel_fro(out["y"].cpu().double().numpy()[rows], ref["y"]) <= TOL_Y[w.dtype]
    # all tokens: routing outputs are consistent with the gate output
    idx_all = out["idx"].cpu().numpy()
    G_all = out["G"].cpu().double().numpy()
    assert np.all(np.abs(G_all.sum(1) - 1.0) <= 1e-5)
    assert all(len(set(r)) == w.k for r in idx_all[:: max(1, w.T // 2048)].tolist())
    if w.groups:
        m = w.n // w.groups
        grp = idx_all // m
        assert np.all(grp.reshape(w.T, w.k_groups, -1).min(2) == grp.reshape(w.T, w.k_groups, -1).max(2))
    check_routing_properties(w, idx_all, G_all, out["counts"].cpu().numpy(),
                             out["importance"].cpu().numpy(), out["cv2"].item())
    # the component calls reproduce the fused call and expose perm / offsets
    r = run_components(w, dinp, ws)
    assert torch.equal(r["y"], out["y"]) and torch.equal(r["idx"], out["idx"])
    check_routing_properties(w, idx_all, G_all, r["counts"].cpu().numpy(),
                             r["importance"].cpu().numpy(), r["cv2"].item(),
                             r["offsets"].cpu().numpy(), r["perm"].cpu().numpy(),
                             r["inv_perm"].cpu().numpy())
