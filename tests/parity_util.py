"""Helpers for the GPU parity tests: run the C-ABI path on device copies of
seeded inputs and compare with the CPU oracle at the stated tolerances.

Tolerances (from the layer's specification): expert indices, counts and the
permutation bit-exact (inputs carry a top-k margin >= 1e-3); gate weights
1e-5 absolute; y 2e-2 relative Frobenius for the bf16 FFN and 1e-4 in fp32
mode; importance 1e-5 relative; CV^2 1e-4 relative.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from oracle.margin import enforce_margin, gate_margins
from sparsely_gated_mixture_top_b300 import binding as B
from sparsely_gated_mixture_top_b300 import workloads as wl

TOL_G = 1e-5
TOL_Y = {"bf16": 2e-2, "f32": 1e-4}
TOL_IMP = 1e-5
TOL_CV2 = 1e-4


def to_dev(inp: dict) -> dict:
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def rel_fro(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a))


def prepared_inputs(w: wl.Workload, rows=None, bg=None):
    """Host inputs with the top-k margin enforced (on `rows`, default all tokens)."""
    inp = wl.make_inputs(w)
    if bg is not None:
        inp["bg"] = bg
    if w.noisy:
        enforce_margin(w, inp, rows)
    return inp


def oracle_full(w: wl.Workload, inp: dict) -> dict:
    return oracle.forward(inp["x"], inp["Wg"], inp["Wn"], inp["bg"], inp["eps"] if w.noisy else None,
                          inp["W1"], inp["b1"], inp["W2"], inp["b2"], w.k, w.groups, w.k_groups)


def check_against_oracle(w: wl.Workload, out: dict, ref: dict, tokens=None) -> None:
    """Compare device outputs with the oracle on all tokens (tokens=None) or on a
    boolean mask of tokens whose top-k choice is unique."""
    idx = out["idx"].cpu().numpy()
    G = out["G"].cpu().double().numpy()
    y = out["y"].cpu().double().numpy()
    sel = slice(None) if tokens is None else tokens
    np.testing.assert_array_equal(idx[sel], ref["idx"][sel])
    assert np.max(np.abs(G[sel] - ref["G"][sel]), initial=0.0) <= TOL_G
    assert rel_fro(y[sel], ref["y"][sel]) <= TOL_Y[w.dtype], rel_fro(y[sel], ref["y"][sel])
    if tokens is None:
        np.testing.assert_array_equal(out["counts"].cpu().numpy(), ref["counts"])
        imp = out["importance"].cpu().double().numpy()
        np.testing.assert_allclose(imp, ref["importance"], rtol=TOL_IMP, atol=TOL_IMP)
        cv2 = float(out["cv2"].cpu().item())
        assert abs(cv2 - ref["cv2"]) <= TOL_CV2 * max(abs(ref["cv2"]), 1e-6)


def check_routing_properties(w: wl.Workload, idx, G, counts, importance, cv2, offsets=None,
                             perm=None, inv_perm=None) -> None:
    """Properties of the routing outputs that hold at any size, given the gate output."""
    idx = np.asarray(idx).reshape(-1)
    G = np.asarray(G, dtype=np.float64).reshape(-1)
    assert idx.min(initial=0) >= 0 and idx.max(initial=0) < w.n
    ref_counts = np.bincount(idx, minlength=w.n)
    np.testing.assert_array_equal(np.asarray(counts), ref_counts)
    ref_imp = np.bincount(idx, weights=G, minlength=w.n)
    np.testing.assert_allclose(np.asarray(importance, dtype=np.float64), ref_imp, rtol=TOL_IMP,
                               atol=TOL_IMP)
    mean = ref_imp.mean()
    ref_cv2 = ref_imp.var() / mean ** 2 if mean else 0.0
    assert abs(float(cv2) - ref_cv2) <= TOL_CV2 * max(abs(ref_cv2), 1e-6)
    if offsets is not None:
        np.testing.assert_array_equal(np.asarray(offsets),
                                      np.concatenate([[0], np.cumsum(ref_counts)]))
    if perm is not None:
        np.testing.assert_array_equal(np.asarray(perm), np.argsort(idx, kind="stable"))
    if inv_perm is not None:
        np.testing.assert_array_equal(np.asarray(inv_perm)[np.asarray(perm)], np.arange(idx.size))


def sampled_oracle(w: wl.Workload, inp: dict, rows) -> dict:
    """Oracle gate and output for the given token rows only."""
    rows = np.asarray(rows)
    x = inp["x"][rows]
    eps = inp["eps"][rows] if w.noisy else None
    if w.groups == 0:
        idx, G, _, _ = oracle.gate_flat(x, inp["Wg"], inp["Wn"], inp["bg"], eps, w.k)
    else:
        idx, G, _ = oracle.gate_hier(x, inp["Wg"], inp["Wn"], inp["bg"], eps, w.groups,
                                     w.k_groups, w.k)
    xr = np.repeat(oracle._f64(x), w.k, axis=0)
    E = oracle.expert_rows(xr, idx.reshape(-1), lambda e: inp["W1"][e], inp["b1"],
                           lambda e: inp["W2"][e], inp["b2"])
    y = (E.reshape(len(rows), w.k, w.d) * G[:, :, None]).sum(axis=1)
    return dict(idx=idx, G=G, y=y)


def run_forward(w: wl.Workload, dinp: dict):
    s = B.shape_of(w)
    ws = B.workspace(s)
    out = B.forward(s, dinp, ws=ws)
    status = B.moe_check(ws)
    assert status == B.MOE_OK, (B.status_string(status), B.error_detail(ws))
    return out, ws


def run_components(w: wl.Workload, dinp: dict, ws=None) -> dict:
    """gate -> dispatch -> expert_ffn -> combine through the four component calls."""
    s = B.shape_of(w)
    ws = B.workspace(s) if ws is None else ws
    dev = dinp["x"].device
    T, k, n, S = w.T, w.k, w.n, w.T * w.k
    dt = dinp["x"].dtype
    r = dict(idx=torch.empty((T, k), dtype=torch.int32, device=dev),
             G=torch.empty((T, k), dtype=torch.float32, device=dev),
             counts=torch.empty(n, dtype=torch.int32, device=dev),
             offsets=torch.empty(n + 1, dtype=torch.int32, device=dev),
             perm=torch.empty(S, dtype=torch.int32, device=dev),
             inv_perm=torch.empty(S, dtype=torch.int32, device=dev),
             importance=torch.empty(n, dtype=torch.float32, device=dev),
             cv2=torch.empty(1, dtype=torch.float32, device=dev),
             Y=torch.empty((S, w.d), dtype=dt, device=dev),
             y=torch.empty((T, w.d), dtype=dt, device=dev))
    B.moe_gate(s, dinp["x"], dinp["Wg"], dinp["Wn"], dinp["bg"], dinp["eps"], r["idx"], r["G"], ws)
    B.moe_dispatch(s, r["idx"], r["G"], r["counts"], r["offsets"], r["perm"], r["inv_perm"],
                   r["importance"], r["cv2"], ws)
    B.moe_expert_ffn(s, dinp["x"], r["perm"], r["offsets"], dinp["W1"], dinp["b1"], dinp["W2"],
                     dinp["b2"], r["Y"], ws)
    B.moe_combine(s, r["Y"], r["inv_perm"], r["G"], r["y"], ws)
    status = B.moe_check(ws)
    assert status == B.MOE_OK, (B.status_string(status), B.error_detail(ws))
    return r
