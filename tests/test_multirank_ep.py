"""The expert-parallel layer (sparsely_gated_mixture_top_b300.expert_parallel)
on CPU ranks: gloo process groups of 2 and 4 spawned processes on 127.0.0.1,
the per-rank steps done by the fp64 oracle (tests/ep_util.OracleOps), the
exchange by the layer's own all-to-all calls.

Experts are split in contiguous blocks over the ranks, every rank gates its
own (ragged, possibly empty) share of the tokens, and the results must equal
the oracle's single-process forward pass over all the tokens: idx and the
per-expert counts exactly, y, G and the merged importance and CV^2 to fp64
rounding; every rank's experts run exactly on the rows routed to them.
("Outrageously Large Neural Networks - 中文验证版", sections 计算设置 and
方法适配: experts spread over devices, batches merged at the MoE layer.)
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))

CASES = {
    "flat_p2": dict(P=2, split=[37, 53], w=dict(T=90, d=64, h=128, n=8, k=2, seed=301,
                                                 bias_std=0.1)),
    "flat_p4_empty_rank": dict(P=4, split=[10, 30, 0, 50],
                               w=dict(T=90, d=64, h=128, n=8, k=2, seed=302, bias_std=0.1)),
    "hier_p2": dict(P=2, split=[41, 23], w=dict(T=64, d=64, h=64, n=16, k=4, groups=4,
                                                k_groups=2, seed=303, bias_std=0.1)),
    "flat_p4_k1": dict(P=4, split=[25, 25, 25, 25],
                       w=dict(T=100, d=64, h=64, n=8, k=1, seed=304, noisy=False)),
}


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(case):
    from sparsely_gated_mixture_top_b300 import workloads as wl
    w = wl.Workload("ep", **case["w"])
    return w, wl.make_inputs(w)


def _rank_main(rank, world, port, name, results):
    for p in (ROOT, TESTS):
        if p not in sys.path:
            sys.path.insert(0, p)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from ep_util import OracleOps, f64, local_experts, shape_ns
        from sparsely_gated_mixture_top_b300.expert_parallel import ExpertParallelMoE
        case = CASES[name]
        w, inp = _inputs(case)
        bounds = np.concatenate([[0], np.cumsum(case["split"])])
        sl = slice(int(bounds[rank]), int(bounds[rank + 1]))
        fields = dict(d=w.d, h=w.h, n=w.n, k=w.k, groups=w.groups, k_groups=w.k_groups,
                      dtype=w.dtype, noisy=w.noisy)
        layer = ExpertParallelMoE(fields, shape_ns, ops=OracleOps())
        W1, b1, W2, b2 = local_experts(inp, layer.first_expert, layer.n_local)
        eps = None if inp["eps"] is None else f64(inp["eps"][sl])
        out = layer.forward(f64(inp["x"][sl]), f64(inp["Wg"]), f64(inp["Wn"]), f64(inp["bg"]),
                            eps, f64(W1), f64(b1), f64(W2), f64(b2))
        results[rank] = {k: (v.numpy() if isinstance(v, torch.Tensor) else v)
                         for k, v in out.items()}
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name", list(CASES))
def test_expert_parallel_matches_single_process_oracle(name):
    import oracle
    case = CASES[name]
    P = case["P"]
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    procs = [ctx.Process(target=_rank_main, args=(r, P, port, name, results)) for r in range(P)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    w, inp = _inputs(case)
    ref = oracle.forward(inp["x"], inp["Wg"], inp["Wn"], inp["bg"], inp["eps"], inp["W1"],
                         inp["b1"], inp["W2"], inp["b2"], w.k, w.groups, w.k_groups)
    bounds = np.concatenate([[0], np.cumsum(case["split"])])
    nl = w.n // P
    for r in range(P):
        got = results[r]
        sl = slice(int(bounds[r]), int(bounds[r + 1]))
        np.testing.assert_array_equal(got["idx"], ref["idx"][sl])
        np.testing.assert_allclose(got["G"], ref["G"][sl], rtol=0, atol=1e-15)
        np.testing.assert_allclose(got["y"], ref["y"][sl], rtol=1e-12, atol=1e-12)
        np.testing.assert_array_equal(got["counts"], np.bincount(ref["idx"][sl].ravel(),
                                                                 minlength=w.n))
        np.testing.assert_allclose(got["importance"], ref["importance"], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(float(np.ravel(got["cv2"])[0]), ref["cv2"], rtol=1e-10)
        # rank r's experts ran on exactly the rows all ranks routed to them
        assert got["rows_in"] == int(ref["counts"][r * nl:(r + 1) * nl].sum())


def test_split_sizes():
    from sparsely_gated_mixture_top_b300.expert_parallel import split_sizes
    counts = np.array([1, 2, 3, 4, 5, 6], np.int32)        # P = 3, two experts each
    recv = np.array([0, 7, 1, 1, 2, 0], np.int32)
    assert split_sizes(counts, recv, 3) == ([3, 7, 11], [7, 2, 2])
