"""The expert-parallel layer's device calls (include/moe_ep.h) and the layer
itself on one GPU.

- moe_ep_regroup against the oracle's merged order (oracle.ep_regroup, pinned
  by brute force), bit for bit, over rank counts, empty experts and several
  row blocks; its device error on counts that do not sum to R.
- moe_gather_rows against plain indexing, bit for bit; a row index out of
  range gives a zero row and the device error.
- moe_importance_cv2 against the dispatch's own CV^2 of the same vector.
- P = 2 and P = 4 ranks driven from one process (tests/ep_util.drive_local:
  each rank's kernels run one after another, the exchange is plain copies,
  nothing waits across ranks) against moe_forward on the whole batch: the
  gate is per token and the expert rows are computed independently of their
  neighbours, so idx, G, counts and y must be identical bit for bit; the
  merged importance within the fp32 bar.
- P = 1 through a one-rank NCCL group (the layer's own all-to-all calls).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

import oracle
from ep_util import drive_local, local_experts
from parity_util import TOL_IMP, TOL_Y, oracle_full, prepared_inputs, rel_fro, run_forward, to_dev
from sparsely_gated_mixture_top_b300 import binding as B
from sparsely_gated_mixture_top_b300 import workloads as wl
from sparsely_gated_mixture_top_b300.expert_parallel import ExpertParallelMoE

pytestmark = pytest.mark.gpu

REGROUP = [
    (1, 8, 0, 50),
    (2, 4, 1, 40),
    (4, 16, 2, 300),
    (8, 32, 3, 700),        # 64 rows per (rank, expert): ~180K rows, 44 row blocks
    (8, 512, 4, 9),         # the 4096-segment limit
    (3, 5, 5, 0),           # nothing received
]


@pytest.mark.parametrize("P,nl,seed,mean", REGROUP)
def test_regroup_matches_oracle(P, nl, seed, mean):
    rng = np.random.default_rng(seed)
    counts = rng.poisson(mean, (P, nl)).astype(np.int32) if mean else np.zeros((P, nl), np.int32)
    if mean:
        counts[rng.random((P, nl)) < 0.2] = 0                 # empty segments
    R = int(counts.sum())
    ws = B.workspace(B.make_shape(1, 64, 64, 1, 1, noisy=False))
    dc = torch.from_numpy(counts.reshape(-1)).cuda()
    off = torch.full((nl + 1,), -7, dtype=torch.int32, device="cuda")
    perm = torch.full((max(R, 1),), -7, dtype=torch.int32, device="cuda")
    inv = torch.full((max(R, 1),), -7, dtype=torch.int32, device="cuda")
    B.moe_ep_regroup(P, nl, dc, R, off, perm, inv, ws)
    assert B.moe_check(ws) == B.MOE_OK
    r_off, r_perm, r_inv = oracle.ep_regroup(counts)
    np.testing.assert_array_equal(off.cpu().numpy(), r_off)
    np.testing.assert_array_equal(perm[:R].cpu().numpy(), r_perm)
    np.testing.assert_array_equal(inv[:R].cpu().numpy(), r_inv)


def test_regroup_errors():
    ws = B.workspace(B.make_shape(1, 64, 64, 1, 1, noisy=False))
    counts = torch.tensor([3, 1, 2, 0], dtype=torch.int32, device="cuda")
    off = torch.empty(3, dtype=torch.int32, device="cuda")
    perm = torch.empty(8, dtype=torch.int32, device="cuda")
    inv = torch.empty(8, dtype=torch.int32, device="cuda")
    B.moe_ep_regroup(2, 2, counts, 7, off, perm, inv, ws)           # the counts sum to 6
    assert B.moe_check(ws) == B.MOE_ERR_DEVICE
    bad = torch.tensor([3, -1, 2, 2], dtype=torch.int32, device="cuda")
    B.moe_ep_regroup(2, 2, bad, 6, off, perm, inv, ws)
    assert B.moe_check(ws) == B.MOE_ERR_DEVICE
    with pytest.raises(B.MoEError) as e:
        B.moe_ep_regroup(8, 513, counts, 6, off, perm, inv, ws)
    assert e.value.status == B.MOE_ERR_UNSUPPORTED
    with pytest.raises(B.MoEError) as e:
        B.moe_ep_regroup(0, 2, counts, 6, off, perm, inv, ws)
    assert e.value.status == B.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("dtype,d,div", [(torch.bfloat16, 512, 4), (torch.float32, 64, 1),
                                         (torch.bfloat16, 1024, 1)])
def test_gather_rows_bit_exact(dtype, d, div):
    g = torch.Generator().manual_seed(d + div)
    src = torch.randn((777, d), generator=g).to(dtype).cuda()
    rows = torch.randint(0, 777 * div, (5000,), generator=g, dtype=torch.int32).cuda()
    dst = torch.empty((5000, d), dtype=dtype, device="cuda")
    ws = B.workspace(B.make_shape(1, 64, 64, 1, 1, noisy=False))
    B.moe_gather_rows(src, rows, div, dst, ws)
    assert B.moe_check(ws) == B.MOE_OK
    ref = src[rows.long() // div]
    assert torch.equal(dst.view(torch.uint8), ref.view(torch.uint8))


def test_gather_rows_out_of_range_row():
    src = torch.ones((10, 64), dtype=torch.bfloat16, device="cuda")
    rows = torch.tensor([0, 9, 10, -1, 3], dtype=torch.int32, device="cuda")
    dst = torch.full((5, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    ws = B.workspace(B.make_shape(1, 64, 64, 1, 1, noisy=False))
    B.moe_gather_rows(src, rows, 1, dst, ws)
    assert B.moe_check(ws) == B.MOE_ERR_DEVICE
    out = dst.float().cpu()
    assert (out[[0, 1, 4]] == 1).all() and (out[[2, 3]] == 0).all()


def test_importance_cv2_matches_dispatch():
    w = wl.Workload("cv2", T=3000, d=64, h=64, n=300, k=3, seed=81)
    d = to_dev(wl.make_inputs(w))
    out, _ = run_forward(w, d)
    cv2 = torch.empty(1, dtype=torch.float32, device="cuda")
    B.moe_importance_cv2(out["importance"], cv2)
    torch.cuda.synchronize()
    assert cv2.item() == out["cv2"].item()
    imp = out["importance"].double().cpu().numpy()
    assert cv2.item() == pytest.approx(imp.var() / imp.mean() ** 2, rel=1e-5)


EP_CASES = [
    (wl.Workload("ep_flat", T=2048, d=512, h=1024, n=64, k=4, seed=91, bias_std=0.1), 2,
     [1000, 1048]),
    (wl.Workload("ep_flat_p4", T=2048, d=512, h=1024, n=64, k=4, seed=92, bias_std=0.1), 4,
     [700, 0, 900, 448]),
    (wl.Workload("ep_hier_p2", T=1024, d=512, h=1024, n=256, k=4, groups=16, k_groups=2,
                 seed=93), 2, [600, 424]),
    (wl.Workload("ep_single_sm_p2", T=900, d=128, h=384, n=12, k=2, seed=94), 2, [450, 450]),
]


def _fields(w):
    return dict(d=w.d, h=w.h, n=w.n, k=w.k, groups=w.groups, k_groups=w.k_groups, dtype=w.dtype,
                noisy=w.noisy)


@pytest.mark.parametrize("w,P,split", EP_CASES, ids=[c[0].name for c in EP_CASES])
def test_ranks_on_one_gpu_equal_the_fused_layer(w, P, split):
    inp = prepared_inputs(w)
    d = to_dev(inp)
    full, _ = run_forward(w, d)
    layers = [ExpertParallelMoE(_fields(w), B.make_shape, ranks=(P, q)) for q in range(P)]
    bounds = np.concatenate([[0], np.cumsum(split)])
    sl = [slice(int(bounds[q]), int(bounds[q + 1])) for q in range(P)]
    xs = [d["x"][s].contiguous() for s in sl]
    epss = [None if d["eps"] is None else d["eps"][s].contiguous() for s in sl]
    experts = [local_experts(d, L.first_expert, L.n_local) for L in layers]
    experts = [tuple(None if t is None else t.contiguous() for t in e) for e in experts]
    outs = drive_local(layers, xs, (d["Wg"], d["Wn"], d["bg"], epss), experts)
    torch.cuda.synchronize()
    for L in layers:
        L.ops.check()
    nl = w.n // P
    counts_all = full["counts"].cpu().numpy()
    for q in range(P):
        o = outs[q]
        assert torch.equal(o["idx"], full["idx"][sl[q]])
        assert torch.equal(o["G"], full["G"][sl[q]])
        assert torch.equal(o["y"].view(torch.uint8), full["y"][sl[q]].view(torch.uint8))
        assert o["rows_in"] == int(counts_all[q * nl:(q + 1) * nl].sum())
    imp = outs[0]["importance"].double().cpu().numpy()
    np.testing.assert_allclose(imp, full["importance"].double().cpu().numpy(), rtol=TOL_IMP,
                               atol=TOL_IMP)
    ref = oracle_full(w, inp)
    y = torch.cat([o["y"] for o in outs]).double().cpu().numpy()
    assert rel_fro(y, ref["y"]) <= TOL_Y[w.dtype]


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_one_rank_nccl_group_equals_the_fused_layer():
    w = wl.Workload("ep_nccl_p1", T=1536, d=512, h=1024, n=32, k=4, seed=95, bias_std=0.1)
    d = to_dev(prepared_inputs(w))
    full, _ = run_forward(w, d)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(_free_port())
    dist.init_process_group("nccl", rank=0, world_size=1,
                            device_id=torch.device("cuda", torch.cuda.current_device()))
    try:
        layer = ExpertParallelMoE(_fields(w), B.make_shape)
        out = layer.forward(d["x"], d["Wg"], d["Wn"], d["bg"], d["eps"], d["W1"], d["b1"],
                            d["W2"], d["b2"])
        torch.cuda.synchronize()
        layer.ops.check()
    finally:
        dist.destroy_process_group()
    assert torch.equal(out["idx"], full["idx"])
    assert torch.equal(out["y"].view(torch.uint8), full["y"].view(torch.uint8))
    assert torch.equal(out["importance"], full["importance"])
    assert out["cv2"].item() == full["cv2"].item()
    assert out["rows_in"] == w.T * w.k
