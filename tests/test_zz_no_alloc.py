"""moe_dispatch_noalloc: the dispatch step for callers that cannot allocate
device memory, such as code running inside another framework's fixed memory
pool or a plug-in whose host owns every allocation (it keeps its scratch in a
static device array of the library instead of a caller-provided workspace).

Each call is checked against numpy (bincount and stable argsort of the expert
indices: the counts, offsets, permutation and importance that routing must
give) and against moe_dispatch, the workspace-based entry point, on two calls
in a row with different shapes, so that scratch contents left over from the
first call would show up in the second.  A shape whose scratch is exactly the
8 MiB limit is accepted and correct; one a chunk larger is rejected.  This
file is collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from parity_util import TOL_CV2, TOL_IMP, check_routing_properties
from sparsely_gated_mixture_top_b300 import binding as B
from sparsely_gated_mixture_top_b300 import workloads as wl

pytestmark = pytest.mark.gpu


def _routing_inputs(T, n, k, seed):
    # k distinct experts per token: choice j lies in [base + j*q, base + (j+1)*q) mod n
    g = torch.Generator().manual_seed(seed)
    q = n // k
    base = torch.randint(0, n, (T, 1), generator=g)
    idx = ((base + torch.arange(k) * q + torch.randint(0, q, (T, k), generator=g)) % n)
    idx = idx.to(torch.int32)
    G = torch.rand((T, k), generator=g) + 0.05
    G = (G / G.sum(1, keepdim=True)).float()
    return idx.cuda(), G.cuda()


def _outputs(T, n, k):
    S = T * k
    return dict(counts=torch.full((n,), -7, dtype=torch.int32, device="cuda"),
                offsets=torch.full((n + 1,), -7, dtype=torch.int32, device="cuda"),
                perm=torch.full((S,), -7, dtype=torch.int32, device="cuda"),
                inv_perm=torch.full((S,), -7, dtype=torch.int32, device="cuda"),
                importance=torch.full((n,), -7.0, device="cuda"),
                cv2=torch.full((1,), -7.0, device="cuda"))


def _noalloc(s, idx, G, T, n, k):
    got = _outputs(T, n, k)
    B.moe_dispatch_noalloc(s, idx, G, got["counts"], got["offsets"], got["perm"],
                           got["inv_perm"], got["importance"], got["cv2"])
    torch.cuda.synchronize()
    return got


def _check_against_numpy(T, n, k, idx, G, got):
    w = wl.Workload("noalloc", T=T, d=64, h=64, n=n, k=k)
    check_routing_properties(w, idx.cpu().numpy(), G.cpu().numpy(), got["counts"].cpu().numpy(),
                             got["importance"].cpu().numpy(), got["cv2"].item(),
                             got["offsets"].cpu().numpy(), got["perm"].cpu().numpy(),
                             got["inv_perm"].cpu().numpy())


def test_noalloc_dispatch_matches_numpy_and_workspace_dispatch_twice():
    # First call: many slots, few experts; second call: fewer slots, many
    # experts and a different chunk count, reusing the same static scratch.
    for T, n, k, seed in ((20000, 64, 4, 1), (3000, 1000, 2, 2)):
        s = B.make_shape(T, 64, 64, n, k)
        idx, G = _routing_inputs(T, n, k, seed)
        got = _noalloc(s, idx, G, T, n, k)
        _check_against_numpy(T, n, k, idx, G, got)
        ref = _outputs(T, n, k)
        ws = B.workspace(s)
        B.moe_dispatch(s, idx, G, ref["counts"], ref["offsets"], ref["perm"], ref["inv_perm"],
                       ref["importance"], ref["cv2"], ws)
        assert B.moe_check(ws) == B.MOE_OK
        for key in ("counts", "offsets", "perm", "inv_perm"):
            assert torch.equal(got[key], ref[key]), key
        np.testing.assert_allclose(got["importance"].cpu().numpy(),
                                   ref["importance"].cpu().numpy(), rtol=TOL_IMP, atol=TOL_IMP)
        assert abs(got["cv2"].item() - ref["cv2"].item()) <= TOL_CV2 * abs(ref["cv2"].item())


# n = 704 experts and S = 862 full chunks of 1024 slots: 256 + 4*S + 8*862*n
# + 4*n bytes, every term a multiple of 256, is exactly 8 MiB.
_AT_LIMIT = (882688 // 4, 704, 4)


def test_noalloc_dispatch_at_its_scratch_limit():
    T, n, k = _AT_LIMIT
    assert 256 + 4 * T * k + 8 * (T * k // 1024) * n + 4 * n == 8 << 20
    s = B.make_shape(T, 64, 64, n, k)
    idx, G = _routing_inputs(T, n, k, 3)
    got = _noalloc(s, idx, G, T, n, k)
    _check_against_numpy(T, n, k, idx, G, got)


def test_noalloc_dispatch_rejects_shapes_beyond_its_scratch():
    dummy = torch.empty(16, dtype=torch.int32, device="cuda")
    T, n, k = _AT_LIMIT
    # 16 more tokens: one more chunk of slots, past the 8 MiB scratch
    for shape in (B.make_shape(T + 16, 64, 64, n, k), B.make_shape(1 << 20, 64, 64, 64, 4)):
        with pytest.raises(B.MoEError) as e:
            B.moe_dispatch_noalloc(shape, dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy)
        assert e.value.status == B.MOE_ERR_UNSUPPORTED
