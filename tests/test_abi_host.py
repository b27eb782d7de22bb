"""Host-side checks of the C ABI (no GPU): the library loads, exports every
entry point include/moe.h declares, validates shapes, sizes workspaces and
rejects bad arguments synchronously before any device work."""
import ctypes
import os
import re

import pytest

from sparsely_gated_mixture_top_b300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", txt)
    return sorted(set(names))


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert len(names) >= 11
    lib = ctypes.CDLL(B.LIB_PATH)
    for name in names:
        assert hasattr(lib, name), name
    assert set(B.EXPORTS) <= set(names)


def test_version_and_status_strings():
    assert B.lib.moe_version() >= 100
    assert B.lib.moe_last_cuda_error() == 0              # no CUDA call has failed
    assert B.lib.moe_cuda_error_name(1).decode() == "cudaErrorInvalidValue"
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert B.status_string(code) and B.status_string(code) != "unknown status"
    assert B.status_string(42) == "unknown status"


GOOD = dict(T=100, d=512, h=1024, n=16, k=4)


@pytest.mark.parametrize("kw,code", [
    (dict(), B.MOE_OK),
    (dict(T=0), B.MOE_OK),
    (dict(T=-1), B.MOE_ERR_INVALID_ARG),
    (dict(k=0), B.MOE_ERR_INVALID_ARG),
    (dict(k=17, n=32), B.MOE_ERR_UNSUPPORTED),
    (dict(k=20, n=16), B.MOE_ERR_INVALID_ARG),          # k > n
    (dict(d=500), B.MOE_ERR_UNSUPPORTED),               # d % 64
    (dict(h=1000), B.MOE_ERR_UNSUPPORTED),
    (dict(dtype=7), B.MOE_ERR_INVALID_ARG),
    (dict(groups=4, k_groups=2), B.MOE_OK),
    (dict(groups=3, k_groups=1), B.MOE_ERR_INVALID_ARG),  # 16 % 3
    (dict(groups=4, k_groups=3), B.MOE_ERR_INVALID_ARG),  # 4 % 3
    (dict(groups=4, k_groups=0), B.MOE_ERR_INVALID_ARG),
    (dict(groups=16, k_groups=2), B.MOE_ERR_INVALID_ARG),  # k/kg = 2 > m = 1
    (dict(groups=0, k_groups=1), B.MOE_ERR_INVALID_ARG),
    (dict(n=20000, k=4), B.MOE_ERR_UNSUPPORTED),         # gate columns
    (dict(T=2 ** 30), B.MOE_ERR_UNSUPPORTED),            # slots overflow int32
])
def test_validate(kw, code):
    args = dict(GOOD)
    args.update(kw)
    dtype = args.pop("dtype", "bf16")
    s = B.make_shape(dtype=dtype, **args)
    assert B.validate(s) == code
    nbytes = B.workspace_bytes(s)
    assert (nbytes > 0) == (code == B.MOE_OK)


def test_workspace_grows_with_tokens():
    a = B.workspace_bytes(B.make_shape(**dict(GOOD, T=10)))
    b = B.workspace_bytes(B.make_shape(**dict(GOOD, T=1000)))
    assert 0 < a < b and a % 256 == 0 and b % 256 == 0


def _fake(addr):
    return ctypes.c_void_p(addr)


def test_bad_pointers_rejected_before_any_launch():
    s = B.make_shape(**GOOD)
    n = B.workspace_bytes(s)
    ok, mis = _fake(1 << 20), _fake((1 << 20) + 8)
    lib = B.lib
    # misaligned x
    assert lib.moe_gate(ctypes.byref(s), mis, ok, ok, None, ok, ok, ok, ok, n, None) == B.MOE_ERR_INVALID_ARG
    # noisy gate without eps
    assert lib.moe_gate(ctypes.byref(s), ok, ok, ok, None, None, ok, ok, ok, n, None) == B.MOE_ERR_INVALID_ARG
    # workspace too small / misaligned / missing
    assert lib.moe_gate(ctypes.byref(s), ok, ok, ok, None, ok, ok, ok, ok, n - 256, None) == B.MOE_ERR_WORKSPACE
    assert lib.moe_gate(ctypes.byref(s), ok, ok, ok, None, ok, ok, ok, mis, n, None) == B.MOE_ERR_WORKSPACE
    assert lib.moe_forward(ctypes.byref(s), ok, ok, ok, None, ok, ok, None, ok, None, ok, ok, ok,
                           None, None, None, None, n, None) == B.MOE_ERR_WORKSPACE
    # missing outputs
    assert lib.moe_dispatch(ctypes.byref(s), ok, ok, None, ok, ok, ok, ok, ok, ok, n, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_expert_ffn(ctypes.byref(s), ok, ok, ok, None, None, ok, None, ok, ok, n, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(ctypes.byref(s), ok, ok, ok, None, ok, n, None) == B.MOE_ERR_INVALID_ARG
    # invalid shape wins over everything
    bad = B.make_shape(**dict(GOOD, k=0))
    assert lib.moe_forward(ctypes.byref(bad), ok, ok, ok, None, ok, ok, None, ok, None, ok, ok, ok,
                           None, None, None, ok, n, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_check(mis, None) == B.MOE_ERR_WORKSPACE
    assert lib.moe_workspace_init(mis, n, None) == B.MOE_ERR_WORKSPACE


def test_backward_rejects_bad_arguments_before_any_launch():
    s = B.make_shape(**GOOD)
    n = B.backward_workspace_bytes(s)
    assert n > 0 and n % 256 == 0
    ok, mis = _fake(1 << 20), _fake((1 << 20) + 8)
    lib = B.lib

    def call(shape=s, x=ok, Wg=ok, Wn=ok, eps=ok, W1=ok, b1=None, W2=ok, b2=None, idx=ok, G=ok,
             imp=ok, dy=ok, w=0.5, dx=ok, dWg=ok, dWn=ok, dbg=None, dW1=ok, db1=None, dW2=ok,
             db2=None, ws=ok, nbytes=n):
        return lib.moe_backward(ctypes.byref(shape), x, Wg, Wn, eps, W1, b1, W2, b2, idx, G, imp,
                                dy, w, dx, dWg, dWn, dbg, dW1, db1, dW2, db2, ws, nbytes, None)

    assert call(x=mis) == B.MOE_ERR_INVALID_ARG
    assert call(dy=None) == B.MOE_ERR_INVALID_ARG
    assert call(dWn=None) == B.MOE_ERR_INVALID_ARG            # noisy shape needs dWnoise
    assert call(eps=None) == B.MOE_ERR_INVALID_ARG
    assert call(imp=None) == B.MOE_ERR_INVALID_ARG            # w_importance != 0 needs importance
    assert call(w=float("nan")) == B.MOE_ERR_INVALID_ARG
    assert call(nbytes=n - 256) == B.MOE_ERR_WORKSPACE
    assert call(ws=mis) == B.MOE_ERR_WORKSPACE
    # the hierarchical gate has a backward too: its workspace adds the routed
    # (token, group) pairs and the transposes of all groups + n score columns
    hier = B.make_shape(**dict(GOOD, n=16, groups=4, k_groups=2, k=4))
    hb = B.backward_workspace_bytes(hier)
    assert hb > n and hb % 256 == 0
    assert call(shape=hier) == B.MOE_ERR_WORKSPACE         # the flat shape's workspace is short
    assert call(shape=B.make_shape(**dict(GOOD, k=0))) == B.MOE_ERR_INVALID_ARG


def test_balanced_rejects_bad_arguments_before_any_launch():
    s = B.make_shape(**GOOD)                    # T=100, n=16, k=4: m = 25, n*m = 400
    cap = 400
    n = B.balanced_workspace_bytes(s, cap)
    assert n > 0 and n % 256 == 0
    assert B.balanced_workspace_bytes(s, 2 * cap) > n
    ok, mis = _fake(1 << 20), _fake((1 << 20) + 8)
    lib = B.lib

    def call(shape=s, x=ok, Wg=ok, Wn=ok, bg=None, eps=ok, thr=None, rows=cap, W1=ok, W2=ok,
             y=ok, counts=ok, W=None, ws=ok, nbytes=n):
        return lib.moe_forward_balanced(ctypes.byref(shape), x, Wg, Wn, bg, eps, thr, rows, W1,
                                        None, W2, None, y, counts, W, ws, nbytes, None)

    assert call(x=mis) == B.MOE_ERR_INVALID_ARG
    assert call(counts=None) == B.MOE_ERR_INVALID_ARG
    assert call(eps=None) == B.MOE_ERR_INVALID_ARG              # noisy shape needs eps
    assert call(rows=cap - 1, nbytes=B.balanced_workspace_bytes(s, cap - 1)) == B.MOE_ERR_INVALID_ARG
    assert call(nbytes=n - 256) == B.MOE_ERR_WORKSPACE
    assert call(ws=mis) == B.MOE_ERR_WORKSPACE
    assert call(rows=-1) == B.MOE_ERR_UNSUPPORTED
    hier = B.make_shape(**dict(GOOD, n=16, groups=4, k_groups=2, k=4))
    assert B.balanced_workspace_bytes(hier, cap) == 0
    assert call(shape=hier) == B.MOE_ERR_UNSUPPORTED
