"""Load estimate of the noisy gate on the GPU (moe_gate_load through the C
ABI) against the CPU oracle.

Tolerance: c and H are fp32-faithful (split-bf16 scores, error ~1e-6) and the
noise scale uses the hardware exp/log (error below 1e-6), so each P(t, i) is
within a few 1e-6 of the oracle for noise scales near 1 and the per-token
errors average out over the sum: load within 1e-4 relative + 1e-3 absolute,
CV^2 within 1e-3 relative.  The gate outputs (idx, G) are also checked.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL_G, prepared_inputs, to_dev
from sparsely_gated_mixture_top_b300 import binding as B
from sparsely_gated_mixture_top_b300 import workloads as wl

pytestmark = pytest.mark.gpu

W = wl.Workload
CASES = [
    W("load_small", T=300, d=128, h=64, n=16, k=2, bias_std=0.1, seed=41),
    W("load_ragged_n70_k3", T=517, d=192, h=64, n=70, k=3, seed=42),
    W("load_k15", T=200, d=64, h=64, n=16, k=15, seed=43),
    W("load_one_expert_kept", T=64, d=64, h=64, n=9, k=1, seed=44),
]


def _run(w, dinp):
    s = B.shape_of(w)
    ws = B.workspace(s)
    lws = torch.empty(B.load_workspace_bytes(s), dtype=torch.uint8, device="cuda")
    idx = torch.empty((w.T, w.k), dtype=torch.int32, device="cuda")
    G = torch.empty((w.T, w.k), dtype=torch.float32, device="cuda")
    load = torch.full((w.n,), -1.0, device="cuda")
    cv2 = torch.full((1,), -1.0, device="cuda")
    B.moe_gate_load(s, dinp["x"], dinp["Wg"], dinp["Wn"], dinp["bg"], dinp["eps"], idx, G, load,
                    cv2, ws, lws)
    assert B.moe_check(ws) == B.MOE_OK
    return idx, G, load, cv2


def _check(w, inp, idx, G, load, cv2):
    P, ref_load, ref_cv2 = oracle.load(inp["x"], inp["Wg"], inp["Wn"], inp["bg"], inp["eps"], w.k)
    ridx, rG, _, _ = oracle.gate_flat(inp["x"], inp["Wg"], inp["Wn"], inp["bg"], inp["eps"], w.k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    assert np.abs(G.cpu().double().numpy() - rG).max() <= TOL_G
    got = load.cpu().double().numpy()
    assert np.all(np.abs(got - ref_load) <= 1e-4 * np.abs(ref_load) + 1e-3), \
        np.abs(got - ref_load).max()
    assert abs(cv2.item() - ref_cv2) <= 1e-3 * max(ref_cv2, 1e-6)


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_load_matches_oracle(w):
    inp = prepared_inputs(w)
    idx, G, load, cv2 = _run(w, to_dev(inp))
    _check(w, inp, idx, G, load, cv2)


def test_load_full_size_flat_workload():
    w = wl.WORKLOADS["flat_n256_k4"]
    inp = prepared_inputs(w)
    idx, G, load, cv2 = _run(w, to_dev(inp))
    _check(w, inp, idx, G, load, cv2)
    # every token contributes at least its k kept experts' mass near the top
    assert load.sum().item() > 0.5 * w.T * w.k


def test_load_unsupported_shapes_are_rejected():
    dummy = torch.empty(64, dtype=torch.float32, device="cuda")
    for kw in (dict(groups=4, k_groups=2, n=16, k=4), dict(dtype="f32"), dict(noisy=False),
               dict(k=16, n=32)):
        base = dict(T=8, d=64, h=64, n=8, k=2)
        base.update(kw)
        s = B.make_shape(**base)
        assert B.load_workspace_bytes(s) == 0
        with pytest.raises(B.MoEError) as e:
            B.moe_gate_load(s, dummy, dummy, dummy, None, dummy, dummy, dummy, dummy, dummy,
                            torch.empty(1 << 20, dtype=torch.uint8, device="cuda"),
                            torch.empty(256, dtype=torch.uint8, device="cuda"))
        assert e.value.status == B.MOE_ERR_UNSUPPORTED
