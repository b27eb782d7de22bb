"""Python binding of the C ABI in include/moe.h (ctypes; argument marshalling only).

Every function here passes torch CUDA tensors' device pointers and sizes to
the shared library `libmoe_b300.so` built in-tree by
`python -m sparsely_gated_mixture_top_b300.build`; every step of the layer
runs in that library's CUDA kernels.  PyTorch supplies device memory and
streams only.  There is no fallback: if the library is missing, importing
this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_b300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_WORKSPACE = -3
MOE_ERR_CUDA = -4
MOE_ERR_TIMEOUT = -5
MOE_ERR_DEVICE = -6
MOE_F32 = 0
MOE_BF16 = 1

EXPORTS = ("moe_version", "moe_status_string", "moe_last_cuda_error", "moe_cuda_error_name",
           "moe_validate", "moe_workspace_bytes",
           "moe_workspace_init", "moe_gate", "moe_dispatch", "moe_expert_ffn", "moe_combine",
           "moe_forward", "moe_check", "moe_dispatch_noalloc", "moe_load_workspace_bytes",
           "moe_gate_load", "moe_backward_workspace_bytes", "moe_backward",
           "moe_balanced_workspace_bytes", "moe_forward_balanced", "moe_selftest_timeout",
           "moe_ep_regroup", "moe_gather_rows", "moe_importance_cv2")


class MoEShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int32), ("h", ctypes.c_int32),
                ("n", ctypes.c_int32), ("k", ctypes.c_int32), ("groups", ctypes.c_int32),
                ("k_groups", ctypes.c_int32), ("dtype", ctypes.c_int32), ("noisy", ctypes.c_int32)]


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = f"{fn}: {status_string(status)} ({status})"
        if status == MOE_ERR_CUDA:
            code = lib.moe_last_cuda_error()
            msg += f" [{lib.moe_cuda_error_name(code).decode()} = {code}]"
        super().__init__(msg)


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run "
                          "`python -m sparsely_gated_mixture_top_b300.build` first")
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz, i32, shp = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.POINTER(MoEShape)
    lib.moe_version.argtypes, lib.moe_version.restype = [], i32
    lib.moe_status_string.argtypes, lib.moe_status_string.restype = [i32], ctypes.c_char_p
    lib.moe_last_cuda_error.argtypes, lib.moe_last_cuda_error.restype = [], i32
    lib.moe_cuda_error_name.argtypes, lib.moe_cuda_error_name.restype = [i32], ctypes.c_char_p
    lib.moe_validate.argtypes, lib.moe_validate.restype = [shp], i32
    lib.moe_workspace_bytes.argtypes, lib.moe_workspace_bytes.restype = [shp], sz
    lib.moe_workspace_init.argtypes, lib.moe_workspace_init.restype = [vp, sz, vp], i32
    lib.moe_gate.argtypes = [shp] + [vp] * 8 + [sz, vp]
    lib.moe_dispatch.argtypes = [shp] + [vp] * 9 + [sz, vp]
    lib.moe_expert_ffn.argtypes = [shp] + [vp] * 9 + [sz, vp]
    lib.moe_combine.argtypes = [shp] + [vp] * 5 + [sz, vp]
    lib.moe_forward.argtypes = [shp] + [vp] * 16 + [sz, vp]
    lib.moe_check.argtypes = [vp, vp]
    lib.moe_dispatch_noalloc.argtypes = [shp] + [vp] * 9
    lib.moe_load_workspace_bytes.argtypes, lib.moe_load_workspace_bytes.restype = [shp], sz
    lib.moe_gate_load.argtypes = [shp] + [vp] * 10 + [sz, vp, sz, vp]
    lib.moe_backward_workspace_bytes.argtypes = [shp]
    lib.moe_backward_workspace_bytes.restype = sz
    lib.moe_backward.argtypes = [shp] + [vp] * 12 + [ctypes.c_float] + [vp] * 9 + [sz, vp]
    lib.moe_balanced_workspace_bytes.argtypes = [shp, ctypes.c_int64]
    lib.moe_balanced_workspace_bytes.restype = sz
    lib.moe_forward_balanced.argtypes = [shp] + [vp] * 6 + [ctypes.c_int64] + [vp] * 8 + [sz, vp]
    lib.moe_selftest_timeout.argtypes = [vp, sz, vp]
    i64 = ctypes.c_int64
    lib.moe_ep_regroup.argtypes = [i32, i32, vp, i64, vp, vp, vp, vp, vp]
    lib.moe_gather_rows.argtypes = [vp, i64, vp, i32, i64, i32, i32, vp, vp, vp]
    lib.moe_importance_cv2.argtypes = [vp, i32, vp, vp]
    for f in ("moe_gate", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_forward",
              "moe_check", "moe_dispatch_noalloc", "moe_gate_load", "moe_backward",
              "moe_forward_balanced", "moe_selftest_timeout", "moe_ep_regroup",
              "moe_gather_rows", "moe_importance_cv2"):
        getattr(lib, f).restype = i32
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.moe_status_string(status).decode()


def _p(t):
    """Device pointer of a tensor (None -> NULL)."""
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ok(fn: str, status: int):
    if status != MOE_OK:
        raise MoEError(fn, status)


def make_shape(T, d, h, n, k, groups=0, k_groups=0, dtype="bf16", noisy=True) -> MoEShape:
    dt = {"bf16": MOE_BF16, "f32": MOE_F32}[dtype] if isinstance(dtype, str) else int(dtype)
    return MoEShape(int(T), int(d), int(h), int(n), int(k), int(groups), int(k_groups), dt,
                    1 if noisy else 0)


def shape_of(w) -> MoEShape:
    """The ABI shape of a workload description (anything with the same fields)."""
    return make_shape(w.T, w.d, w.h, w.n, w.k, w.groups, w.k_groups, w.dtype, w.noisy)


def validate(shape: MoEShape) -> int:
    return lib.moe_validate(ctypes.byref(shape))


def workspace_bytes(shape: MoEShape) -> int:
    return lib.moe_workspace_bytes(ctypes.byref(shape))


def workspace(shape: MoEShape, device="cuda", stream=None) -> torch.Tensor:
    """A fresh workspace (uint8 device tensor) with its error word cleared."""
    nbytes = workspace_bytes(shape)
    if nbytes == 0:
        raise MoEError("moe_workspace_bytes", validate(shape))
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    _ok("moe_workspace_init", lib.moe_workspace_init(_p(ws), nbytes, _stream(stream)))
    return ws


def moe_gate(shape, x, Wg, Wn, bg, eps, idx, G, ws, stream=None):
    _ok("moe_gate", lib.moe_gate(ctypes.byref(shape), _p(x), _p(Wg), _p(Wn), _p(bg), _p(eps),
                                 _p(idx), _p(G), _p(ws), ws.numel(), _stream(stream)))


def moe_dispatch(shape, idx, G, counts, offsets, perm, inv_perm, importance, cv2, ws,
                 stream=None):
    _ok("moe_dispatch", lib.moe_dispatch(ctypes.byref(shape), _p(idx), _p(G), _p(counts),
                                         _p(offsets), _p(perm), _p(inv_perm), _p(importance),
                                         _p(cv2), _p(ws), ws.numel(), _stream(stream)))


def moe_dispatch_noalloc(shape, idx, G, counts, offsets, perm, inv_perm, importance, cv2,
                         stream=None):
    """moe_dispatch for callers that cannot allocate: the routing scratch lives in a
    fixed 8 MiB static device array inside the library (no workspace argument).
    Calls that overlap on the GPU share that array and must be serialised."""
    _ok("moe_dispatch_noalloc", lib.moe_dispatch_noalloc(
        ctypes.byref(shape), _p(idx), _p(G), _p(counts), _p(offsets), _p(perm), _p(inv_perm),
        _p(importance), _p(cv2), _stream(stream)))


def load_workspace_bytes(shape: MoEShape) -> int:
    return lib.moe_load_workspace_bytes(ctypes.byref(shape))


def moe_gate_load(shape, x, Wg, Wn, bg, eps, idx, G, load, load_cv2, ws, lws, stream=None):
    """Gate plus the load estimate of the noisy gate (flat, noisy, bf16)."""
    _ok("moe_gate_load", lib.moe_gate_load(
        ctypes.byref(shape), _p(x), _p(Wg), _p(Wn), _p(bg), _p(eps), _p(idx), _p(G), _p(load),
        _p(load_cv2), _p(ws), ws.numel(), _p(lws), lws.numel(), _stream(stream)))


def moe_expert_ffn(shape, x, perm, offsets, W1, b1, W2, b2, Y_slot, ws, stream=None):
    _ok("moe_expert_ffn", lib.moe_expert_ffn(ctypes.byref(shape), _p(x), _p(perm), _p(offsets),
                                             _p(W1), _p(b1), _p(W2), _p(b2), _p(Y_slot), _p(ws),
                                             ws.numel(), _stream(stream)))


def moe_combine(shape, Y_slot, inv_perm, G, y, ws, stream=None):
    _ok("moe_combine", lib.moe_combine(ctypes.byref(shape), _p(Y_slot), _p(inv_perm), _p(G),
                                       _p(y), _p(ws), ws.numel(), _stream(stream)))


def moe_forward(shape, x, Wg, Wn, bg, eps, W1, b1, W2, b2, y, G, idx, importance, cv2, counts,
                ws, stream=None):
    _ok("moe_forward", lib.moe_forward(ctypes.byref(shape), _p(x), _p(Wg), _p(Wn), _p(bg),
                                       _p(eps), _p(W1), _p(b1), _p(W2), _p(b2), _p(y), _p(G),
                                       _p(idx), _p(importance), _p(cv2), _p(counts), _p(ws),
                                       ws.numel(), _stream(stream)))


def moe_check(ws, stream=None) -> int:
    """Synchronises the stream; returns (and clears) the workspace's device error code."""
    return lib.moe_check(_p(ws), _stream(stream))


def error_detail(ws) -> tuple[int, int, int]:
    """(code, site, aux) of the workspace's error word, without clearing it."""
    h = ws[:16].view(torch.int32).cpu().tolist()
    return h[0], h[1], h[2]


# --------------------------------------------------------------------------
# Convenience: allocate outputs and run the layer.
# --------------------------------------------------------------------------
def outputs(shape: MoEShape, device="cuda") -> dict:
    dt = torch.bfloat16 if shape.dtype == MOE_BF16 else torch.float32
    T, k, n = shape.T, shape.k, shape.n
    return dict(y=torch.empty((T, shape.d), dtype=dt, device=device),
                G=torch.empty((T, k), dtype=torch.float32, device=device),
                idx=torch.empty((T, k), dtype=torch.int32, device=device),
                importance=torch.empty(n, dtype=torch.float32, device=device),
                cv2=torch.empty(1, dtype=torch.float32, device=device),
                counts=torch.empty(n, dtype=torch.int32, device=device))


def forward(shape: MoEShape, inp: dict, ws=None, out=None, stream=None) -> dict:
    """moe_forward on device tensors inp = {x, Wg, Wn, bg, eps, W1, b1, W2, b2}."""
    dev = inp["x"].device
    ws = workspace(shape, dev, stream) if ws is None else ws
    out = outputs(shape, dev) if out is None else out
    moe_forward(shape, inp["x"], inp["Wg"], inp.get("Wn"), inp.get("bg"), inp.get("eps"),
                inp["W1"], inp.get("b1"), inp["W2"], inp.get("b2"), out["y"], out["G"],
                out["idx"], out["importance"], out["cv2"], out["counts"], ws, stream)
    return out


def backward_workspace_bytes(shape: MoEShape) -> int:
    return lib.moe_backward_workspace_bytes(ctypes.byref(shape))


def backward_workspace(shape: MoEShape, device="cuda", stream=None) -> torch.Tensor:
    """A fresh backward workspace (uint8 device tensor) with its error word cleared."""
    nbytes = backward_workspace_bytes(shape)
    if nbytes == 0:
        raise MoEError("moe_backward_workspace_bytes", validate(shape) or MOE_ERR_UNSUPPORTED)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    _ok("moe_workspace_init", lib.moe_workspace_init(_p(ws), nbytes, _stream(stream)))
    return ws


def moe_backward(shape, x, Wg, Wn, eps, W1, b1, W2, b2, idx, G, importance, dy, w_importance,
                 dx, dWg, dWn, dbg, dW1, db1, dW2, db2, ws, stream=None):
    """Gradients of sum <dy, y> + w_importance * CV^2(importance) (flat layer)."""
    _ok("moe_backward", lib.moe_backward(
        ctypes.byref(shape), _p(x), _p(Wg), _p(Wn), _p(eps), _p(W1), _p(b1), _p(W2), _p(b2),
        _p(idx), _p(G), _p(importance), _p(dy), float(w_importance), _p(dx), _p(dWg), _p(dWn),
        _p(dbg), _p(dW1), _p(db1), _p(dW2), _p(db2), _p(ws), ws.numel(), _stream(stream)))


def balanced_workspace_bytes(shape: MoEShape, rows_cap: int) -> int:
    return lib.moe_balanced_workspace_bytes(ctypes.byref(shape), int(rows_cap))


def balanced_workspace(shape: MoEShape, rows_cap: int, device="cuda", stream=None) -> torch.Tensor:
    """A fresh workspace for moe_forward_balanced with its error word cleared."""
    nbytes = balanced_workspace_bytes(shape, rows_cap)
    if nbytes == 0:
        raise MoEError("moe_balanced_workspace_bytes", validate(shape) or MOE_ERR_UNSUPPORTED)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    _ok("moe_workspace_init", lib.moe_workspace_init(_p(ws), nbytes, _stream(stream)))
    return ws


def moe_forward_balanced(shape, x, Wg, Wn, bg, eps, thr, rows_cap, W1, b1, W2, b2, y, counts, W,
                         ws, stream=None):
    """The layer with balanced routing: thr None = batchwise mask (each expert
    keeps floor(k*T/n) tokens), else per-expert thresholds."""
    _ok("moe_forward_balanced", lib.moe_forward_balanced(
        ctypes.byref(shape), _p(x), _p(Wg), _p(Wn), _p(bg), _p(eps), _p(thr), int(rows_cap),
        _p(W1), _p(b1), _p(W2), _p(b2), _p(y), _p(counts), _p(W), _p(ws), ws.numel(),
        _stream(stream)))


def moe_selftest_timeout(ws, stream=None):
    """Diagnostic: a bounded wait that runs out (MOE_ERR_TIMEOUT in ws after ~2 s)."""
    _ok("moe_selftest_timeout", lib.moe_selftest_timeout(_p(ws), ws.numel(), _stream(stream)))


# --------------------------------------------------------------------------
# Expert-parallel device calls (include/moe_ep.h).  `err` is a workspace (its
# error word is used) or None.
# --------------------------------------------------------------------------
def moe_ep_regroup(P, n_local, recv_counts, R, offsets_local, perm_local, inv_local, err=None,
                   stream=None):
    _ok("moe_ep_regroup", lib.moe_ep_regroup(int(P), int(n_local), _p(recv_counts), int(R),
                                             _p(offsets_local), _p(perm_local), _p(inv_local),
                                             _p(err), _stream(stream)))


def moe_gather_rows(src, rows, div, dst, err=None, stream=None):
    """dst[i] = src[rows[i] // div] (rows of src.shape[1] elements)."""
    dt = {torch.bfloat16: MOE_BF16, torch.float32: MOE_F32}[src.dtype]
    assert dst.dtype == src.dtype and dst.shape[1:] == src.shape[1:] and src.dim() == 2
    _ok("moe_gather_rows", lib.moe_gather_rows(_p(src), src.shape[0], _p(rows), int(div),
                                               dst.shape[0], src.shape[1], dt, _p(dst), _p(err),
                                               _stream(stream)))


def moe_importance_cv2(importance, cv2, stream=None):
    _ok("moe_importance_cv2", lib.moe_importance_cv2(_p(importance), importance.numel(),
                                                     _p(cv2), _stream(stream)))


# --------------------------------------------------------------------------
# CUDA graphs: one layer call recorded once and replayed without per-kernel
# launch cost.  The replay reads and writes the same tensors as the recorded
# call; refill the inputs in place between replays.
# --------------------------------------------------------------------------
def capture(fn) -> torch.cuda.CUDAGraph:
    """Records fn() as a CUDA graph.  fn calls this module's functions with
    stream=None (the capture stream is then the current stream) on tensors
    that exist before the capture; the graph is kept so that its nodes can
    be inspected (kernel_nodes)."""
    g = torch.cuda.CUDAGraph(keep_graph=True)
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        fn()
    return g


def kernel_nodes(g: torch.cuda.CUDAGraph) -> int:
    """The number of kernel launches recorded in a captured graph (memset
    and memcpy nodes are not counted)."""
    from cuda.bindings import runtime as rt
    handle = rt.cudaGraph_t(init_value=g.raw_cuda_graph())
    err, _, num = rt.cudaGraphGetNodes(handle, 0)
    if err != rt.cudaError_t.cudaSuccess:
        raise RuntimeError(f"cudaGraphGetNodes: {err}")
    err, nodes, num = rt.cudaGraphGetNodes(handle, num)
    if err != rt.cudaError_t.cudaSuccess:
        raise RuntimeError(f"cudaGraphGetNodes: {err}")
    kernel = rt.cudaGraphNodeType.cudaGraphNodeTypeKernel
    return sum(1 for nd in nodes[:num] if rt.cudaGraphNodeGetType(nd)[1] == kernel)
