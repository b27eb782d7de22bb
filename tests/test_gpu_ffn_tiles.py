"""The expert stage (moe_expert_ffn, through the C ABI) on expert row counts
chosen to hit every edge of its tiling: experts with 1, 15, 16, 17, 255,
256, 257, 511, 512 and 513 rows, empty experts, and output widths of one and
of several 256-feature blocks ("MoE:稀疏门控混合专家", section 二: each expert
is a one-hidden-layer ReLU network applied to the rows routed to it).

The routing is the oracle's (numpy-pinned) permutation of a token -> expert
assignment built to give those counts; every expert row is compared with the
oracle's expert on that row: the whole stage within the bf16 bar (2e-2
relative Frobenius) and every single row within 5e-2, so that one wrong row
at a tile edge cannot hide in the total.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL_Y, rel_fro
from sparsely_gated_mixture_top_b300 import binding as B
from sparsely_gated_mixture_top_b300 import workloads as wl

pytestmark = pytest.mark.gpu

EDGE_COUNTS = [1, 15, 16, 17, 31, 255, 256, 257, 0, 511, 512, 513, 700, 3, 0, 48]

CASES = [
    ("edges_d256_h512", 256, 512, EDGE_COUNTS),
    ("edges_d512_h1024", 512, 1024, EDGE_COUNTS),
    ("around_256_d512_h1024", 512, 1024, [240, 250, 256, 260, 270, 300, 248, 255, 257, 262]),
    ("narrow_d128_h256", 128, 256, [5, 130, 257, 0, 64]),     # layer 2 on the single-SM kernel
]


def stage(d, h, counts, seed):
    n = len(counts)
    T = int(sum(counts))
    w = wl.Workload("tiles", T=T, d=d, h=h, n=n, k=1, bias_std=0.2, seed=seed)
    inp = wl.make_inputs(w)
    rng = np.random.default_rng(seed)
    idx = rng.permutation(np.repeat(np.arange(n), counts)).astype(np.int32).reshape(T, 1)
    G = np.ones((T, 1))
    c, offsets, perm, inv, _, _ = oracle.route(idx, G, n)
    np.testing.assert_array_equal(c, counts)
    s = B.shape_of(w)
    ws = B.workspace(s)
    Y = torch.full((T, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.moe_expert_ffn(s, inp["x"].cuda(), torch.from_numpy(perm).cuda(),
                     torch.from_numpy(offsets).cuda(), inp["W1"].cuda(), inp["b1"].cuda(),
                     inp["W2"].cuda(), inp["b2"].cuda(), Y, ws)
    assert B.moe_check(ws) == B.MOE_OK
    Yref = oracle.expert_rows(oracle._f64(inp["x"])[perm], idx.reshape(-1)[perm], inp["W1"],
                              inp["b1"], inp["W2"], inp["b2"])
    return Y.cpu().double().numpy(), Yref


@pytest.mark.parametrize("name,d,h,counts", CASES, ids=[c[0] for c in CASES])
def test_expert_stage_on_tile_edges(name, d, h, counts):
    got, ref = stage(d, h, counts, seed=41 + len(name))
    assert np.isfinite(got).all()
    assert rel_fro(got, ref) <= TOL_Y["bf16"]
    row_err = np.linalg.norm(got - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-6)
    assert row_err.max() <= 5e-2, (int(row_err.argmax()), float(row_err.max()))
