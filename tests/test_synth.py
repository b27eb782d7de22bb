"""The seeded input generator: its published mixing function, its distribution,
counter addressing (any slice equals the same slice of the whole tensor) and
its rounding to bf16."""
import math

import numpy as np
import pytest
import torch

from sparsely_gated_mixture_top_b300 import synth, workloads as wl


def test_splitmix64_published_outputs():
    # First outputs of the splitmix64 generator seeded with 0 (Steele, Lea, Flood 2014;
    # the state advances by 0x9E3779B97F4A7C15 and the mixer is applied to it).
    assert synth.splitmix64(0) == 0xE220A8397B1DCDAF
    assert synth.splitmix64(0x9E3779B97F4A7C15) == 0x6E789E6AA1B965F4
    assert synth.splitmix64((2 * 0x9E3779B97F4A7C15) % 2 ** 64) == 0x06C45D188009454F


def test_normal_moments():
    out = torch.empty(1 << 20, dtype=torch.float32)
    synth.fill_normal(out, 1, 2, 0, 0, 1.0)
    a = out.double().numpy()
    assert abs(a.mean()) < 5e-3 and abs(a.var() - 1.0) < 5e-3
    assert abs(np.mean(a ** 3)) < 1e-2 and abs(np.mean(a ** 4) - 3.0) < 3e-2
    assert abs(np.mean(np.abs(a) < 2.0) - 0.9545) < 2e-3     # "mostly within -2..2"


def test_counter_addressing_and_attempts():
    full = torch.empty(1000, dtype=torch.float32)
    synth.fill_normal(full, 9, 5, 0, 0, 1.0)
    part = torch.empty(300, dtype=torch.float32)
    synth.fill_normal(part, 9, 5, 0, 450, 1.0)
    assert torch.equal(full[450:750], part)
    other = torch.empty(300, dtype=torch.float32)
    synth.fill_normal(other, 9, 5, 1, 450, 1.0)
    assert not torch.equal(other, part)


def test_bf16_is_rne_of_the_fp32_value():
    f = torch.empty(1 << 16, dtype=torch.float32)
    b = torch.empty(1 << 16, dtype=torch.bfloat16)
    synth.fill_normal(f, 3, 6, 0, 0, 0.0625)
    synth.fill_normal(b, 3, 6, 0, 0, 0.0625)
    assert torch.equal(f.to(torch.bfloat16), b)       # torch's conversion rounds to nearest even


def test_workload_slices_match_full_tensors():
    w = wl.WORKLOADS["tiny_flat_fp32"].with_(T=40, n=4, bias_std=0.1)
    full = wl.make_inputs(w)
    part = wl.make_inputs(w, experts=False, tokens=slice(10, 25))
    assert torch.equal(part["x"], full["x"][10:25]) and torch.equal(part["eps"], full["eps"][10:25])
    assert torch.equal(wl.expert_weight(w, "W1", 2), full["W1"][2])
    assert torch.equal(wl.expert_weight(w, "W2", 3), full["W2"][3])
    assert torch.equal(wl.expert_bias(w, "b1", 1), full["b1"][1])
    assert torch.equal(wl.eps_rows(w, [7, 3], [0, 0]), full["eps"][[7, 3]])
    assert full["W1"].std().item() == pytest.approx(math.sqrt(2.0 / w.d), rel=0.02)
    assert full["W2"].std().item() == pytest.approx(math.sqrt(1.0 / w.h), rel=0.02)


def test_zipf_gate_bias():
    w = wl.WORKLOADS["skewed_zipf_n64"]
    b = wl.gate_bias(w)
    assert b.shape == (64,)
    assert b[0].item() == 0.0 and b[1].item() == pytest.approx(2 * math.log(0.5), rel=1e-6)
    assert torch.all(b[1:] < b[:-1])


def test_cut_margin_redraws_single_cells():
    """The balanced-routing cut margin redraws single eps cells: afterwards
    every column's cut clears the margin, and a changed cell never moves the
    scores of another column."""
    import oracle
    from oracle.margin import column_cut_gaps, enforce_cut_margin
    w = wl.Workload("cut", T=500, d=32, h=64, n=6, k=2, seed=3)
    inp = wl.make_inputs(w, experts=False)
    before = inp["eps"].clone()
    _, _, H0, _ = oracle.gate_flat(inp["x"], inp["Wg"], inp["Wn"], inp["bg"], inp["eps"], 1)
    ranks = [w.k * w.T // w.n] * w.n
    redraws = enforce_cut_margin(w, inp, ranks, min_margin=5e-3)
    assert redraws > 0
    _, _, H1, _ = oracle.gate_flat(inp["x"], inp["Wg"], inp["Wn"], inp["bg"], inp["eps"], 1)
    assert column_cut_gaps(H1, ranks).min() >= 5e-3
    changed = (inp["eps"] != before).numpy()
    assert changed.sum() >= 1
    np.testing.assert_array_equal(H1[~changed], H0[~changed])
    # the same redraw sequence again gives the same tensor (counter-based draws)
    again = wl.make_inputs(w, experts=False)
    enforce_cut_margin(w, again, ranks, min_margin=5e-3)
    assert torch.equal(again["eps"], inp["eps"])
