"""The layer recorded as a CUDA graph (binding.capture): the replay gives the
eager call's results bit for bit, and the graph holds exactly the kernels the
bench line claims per step (bench.launches_per_step, bench.backward_launches).

Each case runs moe_forward once eagerly, records the same call, refills the
outputs with garbage, replays, and compares every output exactly: the path
is deterministic (fixed-order sums everywhere), so any difference means the
graph dropped or reordered work.
"""
import pytest
import torch

import bench
from parity_util import to_dev
from sparsely_gated_mixture_top_b300 import binding as B
from sparsely_gated_mixture_top_b300 import workloads as wl

pytestmark = pytest.mark.gpu

W = wl.Workload
CASES = [
    W("graph_flat_pair", T=2048, d=512, h=1024, n=64, k=4, seed=71),
    W("graph_flat_single_sm", T=700, d=128, h=384, n=12, k=2, seed=72),
    W("graph_hier", T=1024, d=512, h=1024, n=256, k=4, groups=16, k_groups=2, seed=73),
    W("graph_f32", T=256, d=256, h=512, n=8, k=2, dtype="f32", seed=74),
]
OUTS = ("y", "G", "idx", "importance", "cv2", "counts")


def _call(s, d, out, ws):
    return lambda: B.moe_forward(s, d["x"], d["Wg"], d["Wn"], d["bg"], d["eps"], d["W1"], d["b1"],
                                 d["W2"], d["b2"], out["y"], out["G"], out["idx"],
                                 out["importance"], out["cv2"], out["counts"], ws, None)


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_forward_graph_replays_the_eager_call(w):
    d = to_dev(wl.make_inputs(w))
    s = B.shape_of(w)
    ws = B.workspace(s)
    out = B.outputs(s)
    call = _call(s, d, out, ws)
    call()
    torch.cuda.synchronize()
    assert B.moe_check(ws) == B.MOE_OK
    eager = {k: v.clone() for k, v in out.items()}
    g = B.capture(call)
    assert B.kernel_nodes(g) == bench.launches_per_step(w)
    for v in out.values():
        v.view(torch.uint8).fill_(0xA5)
    g.replay()
    torch.cuda.synchronize()
    assert B.moe_check(ws) == B.MOE_OK
    for k in OUTS:
        assert torch.equal(out[k].view(torch.uint8), eager[k].view(torch.uint8)), k


def test_backward_graph_kernel_count():
    w = W("graph_bwd", T=1024, d=256, h=512, n=16, k=2, seed=75)
    d = to_dev(wl.make_inputs(w))
    s = B.shape_of(w)
    fwd = B.forward(s, d)
    bws = B.backward_workspace(s)
    dev = d["x"].device
    dy = torch.randn((w.T, w.d), generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).to(dev)

    def f32(*shape):
        return torch.empty(shape, dtype=torch.float32, device=dev)

    g = dict(dx=f32(w.T, w.d), dWg=f32(w.d, w.n), dWn=f32(w.d, w.n), dbg=f32(w.n),
             dW1=f32(w.n, w.h, w.d), db1=f32(w.n, w.h), dW2=f32(w.n, w.d, w.h), db2=f32(w.n, w.d))

    def step():
        B.moe_backward(s, d["x"], d["Wg"], d["Wn"], d["eps"], d["W1"], d["b1"], d["W2"], d["b2"],
                       fwd["idx"], fwd["G"], fwd["importance"], dy, 0.01, g["dx"], g["dWg"],
                       g["dWn"], g["dbg"], g["dW1"], g["db1"], g["dW2"], g["db2"], bws, None)

    step()
    torch.cuda.synchronize()
    assert B.moe_check(bws) == B.MOE_OK
    eager = {k: v.clone() for k, v in g.items()}
    graph = B.capture(step)
    assert B.kernel_nodes(graph) == bench.backward_launches(w)
    for v in g.values():
        v.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert B.moe_check(bws) == B.MOE_OK
    for k in g:
        assert torch.equal(g[k], eager[k]), k
