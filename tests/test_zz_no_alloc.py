"""moe_dispatch_noalloc: the dispatch step for callers that cannot allocate
device memory (it keeps its scratch in a static device array of the library
instead of a caller-provided workspace).

Checked against moe_dispatch, the workspace-based entry point, on two calls
in a row with different shapes, so that scratch contents left over from the
first call would show up in the second.  This file is collected last on
purpose: if it fails, a run that stops at the first failure has already run
every other test.
"""
import numpy as np
import pytest
import torch

from parity_util import TOL_CV2, TOL_IMP
from sparsely_gated_mixture_top_b300 import binding as B

pytestmark = pytest.mark.gpu


def _routing_inputs(T, n, k, seed):
    g = torch.Generator().manual_seed(seed)
    idx = torch.stack([torch.randperm(n, generator=g)[:k] for _ in range(T)]).to(torch.int32)
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


def _dispatch_both(T, n, k, seed):
    s = B.make_shape(T, 64, 64, n, k)
    idx, G = _routing_inputs(T, n, k, seed)
    ref, got = _outputs(T, n, k), _outputs(T, n, k)
    ws = B.workspace(s)
    B.moe_dispatch(s, idx, G, ref["counts"], ref["offsets"], ref["perm"], ref["inv_perm"],
                   ref["importance"], ref["cv2"], ws)
    B.moe_dispatch_noalloc(s, idx, G, got["counts"], got["offsets"], got["perm"],
                           got["inv_perm"], got["importance"], got["cv2"])
    torch.cuda.synchronize()
    assert B.moe_check(ws) == B.MOE_OK
    return ref, got


def test_noalloc_dispatch_matches_workspace_dispatch_twice():
    # First call: many slots, few experts; second call: fewer slots, many
    # experts and a different chunk count, reusing the same static scratch.
    for T, n, k, seed in ((20000, 64, 4, 1), (3000, 1000, 2, 2)):
        ref, got = _dispatch_both(T, n, k, seed)
        for key in ("counts", "offsets", "perm", "inv_perm"):
            assert torch.equal(got[key], ref[key]), key
        np.testing.assert_allclose(got["importance"].cpu().numpy(),
                                   ref["importance"].cpu().numpy(), rtol=TOL_IMP, atol=TOL_IMP)
        assert abs(got["cv2"].item() - ref["cv2"].item()) <= TOL_CV2 * abs(ref["cv2"].item())


def test_noalloc_dispatch_rejects_shapes_beyond_its_scratch():
    # 4*S alone exceeds the 8 MiB static scratch.
    s = B.make_shape(1 << 20, 64, 64, 64, 4)
    dummy = torch.empty(16, dtype=torch.int32, device="cuda")
    with pytest.raises(B.MoEError) as e:
        B.moe_dispatch_noalloc(s, dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy)
    assert e.value.status == B.MOE_ERR_UNSUPPORTED
