"""CPU oracle of the MoE layer forward and backward passes (ctypes front of `oracle.c`).

TEST INFRASTRUCTURE ONLY: the tests, the package entry file's smoke check and
the benchmark's CPU-baseline leg may import this module; the product path never
does.  Every function converts its inputs to float64 (exact for bf16/fp32
storage) and calls the plain C implementation in `oracle.c`, which shares no
code with the CUDA path.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/liboracle.so (gcc, OpenMP, no fast-math, no contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
                               "-fPIC", "-shared", "-o", _LIB, _SRC, "-lm"])
    return _LIB


def _lib_():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        i64, i32, vp, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_double
        lib.oracle_softplus.argtypes = [dbl]
        lib.oracle_softplus.restype = dbl
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = i32
        lib.oracle_gate_flat.argtypes = [i64, i32, i32, i32] + [vp] * 9
        lib.oracle_gate_flat.restype = i32
        lib.oracle_gate_hier.argtypes = [i64, i32, i32, i32, i32, i32] + [vp] * 8
        lib.oracle_gate_hier.restype = i32
        lib.oracle_route.argtypes = [i64, i32, i32] + [vp] * 8
        lib.oracle_route.restype = i32
        lib.oracle_expert.argtypes = [i32, i32] + [vp] * 7
        lib.oracle_expert.restype = None
        lib.oracle_experts_combine.argtypes = [i64, i32, i32, i32, i32] + [vp] * 8
        lib.oracle_experts_combine.restype = i32
        lib.oracle_forward.argtypes = [i64, i32, i32, i32, i32, i32, i32] + [vp] * 18
        lib.oracle_forward.restype = i32
        lib.oracle_load.argtypes = [i64, i32, i32, i32] + [vp] * 8
        lib.oracle_load.restype = i32
        lib.oracle_combine_rows.argtypes = [i64, i32, i32, i64] + [vp] * 4
        lib.oracle_combine_rows.restype = i32
        lib.oracle_backward_flat.argtypes = [i64, i32, i32, i32, i32] + [vp] * 10 + [dbl] + [vp] * 10
        lib.oracle_backward_flat.restype = i32
        lib.oracle_forward_balanced.argtypes = [i64, i32, i32, i32, i32] + [vp] * 13
        lib.oracle_forward_balanced.restype = i32
        _lib = lib
    return _lib


def _f64(a):
    """Exact float64 copy of a numpy array or torch tensor (None passes through)."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        import torch
        a = a.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _p(a):
    return None if a is None else a.ctypes.data


def num_threads() -> int:
    return _lib_().oracle_num_threads()


def softplus(z: float) -> float:
    return _lib_().oracle_softplus(float(z))


def gate_flat(x, Wg, Wn, bg, eps, k: int):
    """Flat noisy top-k gate.  Returns idx [T,k] int32, G [T,k], H [T,n], margin [T]."""
    x, Wg, Wn, bg, eps = map(_f64, (x, Wg, Wn, bg, eps))
    T, d = x.shape
    n = Wg.shape[1]
    idx = np.zeros((T, k), np.int32)
    G = np.zeros((T, k))
    H = np.zeros((T, n))
    margin = np.zeros(T)
    rc = _lib_().oracle_gate_flat(T, d, n, k, _p(x), _p(Wg), _p(Wn), _p(bg), _p(eps), _p(idx),
                                  _p(G), _p(H), _p(margin))
    if rc:
        raise ValueError("oracle_gate_flat: bad arguments")
    return idx, G, H, margin


def load(x, Wg, Wn, bg, eps, k: int):
    """Load estimate of the flat noisy gate: P [T,n] (probability that expert i
    stays in the top k when its own noise is redrawn), load [n] = sum over
    tokens, and the CV^2 of load."""
    x, Wg, Wn, bg, eps = map(_f64, (x, Wg, Wn, bg, eps))
    T, d = x.shape
    n = Wg.shape[1]
    P = np.zeros((T, n))
    ld = np.zeros(n)
    cv2 = np.zeros(1)
    rc = _lib_().oracle_load(T, d, n, k, _p(x), _p(Wg), _p(Wn), _p(bg), _p(eps), _p(P), _p(ld),
                             _p(cv2))
    if rc:
        raise ValueError("oracle_load: bad arguments")
    return P, ld, float(cv2[0])


def gate_hier(x, Wg, Wn, bg, eps, groups: int, k_groups: int, k: int):
    """Hierarchical noisy gate.  Returns idx [T,k] int32, G [T,k], margin [T]."""
    x, Wg, Wn, bg, eps = map(_f64, (x, Wg, Wn, bg, eps))
    T, d = x.shape
    n = Wg.shape[1] - groups
    if k % k_groups or n % groups:
        raise ValueError("k must be a multiple of k_groups and n of groups")
    idx = np.zeros((T, k), np.int32)
    G = np.zeros((T, k))
    margin = np.zeros(T)
    rc = _lib_().oracle_gate_hier(T, d, groups, n // groups, k_groups, k // k_groups, _p(x),
                                  _p(Wg), _p(Wn), _p(bg), _p(eps), _p(idx), _p(G), _p(margin))
    if rc:
        raise ValueError("oracle_gate_hier: bad arguments")
    return idx, G, margin


def route(idx, G, n: int):
    """Routing.  Returns counts, offsets, perm, inv_perm, importance, cv2."""
    idx = _i32(idx)
    G = _f64(G)
    T, k = idx.shape
    S = T * k
    counts = np.zeros(n, np.int32)
    offsets = np.zeros(n + 1, np.int32)
    perm = np.zeros(max(S, 1), np.int32)
    inv_perm = np.zeros(max(S, 1), np.int32)
    importance = np.zeros(n)
    cv2 = ctypes.c_double(0.0)
    rc = _lib_().oracle_route(T, n, k, _p(idx), _p(G), _p(counts), _p(offsets), _p(perm),
                              _p(inv_perm), _p(importance), ctypes.addressof(cv2))
    if rc:
        raise ValueError("oracle_route: bad arguments")
    return counts, offsets, perm[:S], inv_perm[:S], importance, cv2.value


def expert(x_row, W1e, b1e, W2e, b2e):
    """E(x) for one token and one expert (W1e [h,d], W2e [d,h])."""
    x_row, W1e, b1e, W2e, b2e = map(_f64, (x_row, W1e, b1e, W2e, b2e))
    h, d = W1e.shape
    a = np.zeros(h)
    out = np.zeros(d)
    _lib_().oracle_expert(d, h, _p(x_row), _p(W1e), _p(b1e), _p(W2e), _p(b2e), _p(a), _p(out))
    return out


def experts_combine(x, idx, G, W1, b1, W2, b2):
    """y[t] = sum_j G[t,j] E_{idx[t,j]}(x_t)."""
    x, G, W1, b1, W2, b2 = map(_f64, (x, G, W1, b1, W2, b2))
    idx = _i32(idx)
    T, d = x.shape
    n, h, _ = W1.shape
    k = idx.shape[1]
    y = np.zeros((T, d))
    rc = _lib_().oracle_experts_combine(T, d, h, n, k, _p(x), _p(idx), _p(G), _p(W1), _p(b1),
                                        _p(W2), _p(b2), _p(y))
    if rc:
        raise ValueError("oracle_experts_combine: bad arguments")
    return y


def combine_rows(Y, inv_perm, G):
    """y[t] = sum_j G[t,j] * Y[inv_perm[t*k+j]] from expert-order rows Y [S, d]."""
    Y, G = _f64(Y), _f64(G)
    inv_perm = _i32(inv_perm)
    T, k = G.shape
    S, d = Y.shape
    y = np.zeros((T, d))
    rc = _lib_().oracle_combine_rows(T, d, k, S, _p(Y), _p(inv_perm), _p(G), _p(y))
    if rc:
        raise ValueError("oracle_combine_rows: bad arguments")
    return y


def expert_rows(x_rows, experts, W1, b1, W2, b2):
    """E_{experts[i]}(x_rows[i]) for each i.  W1/W2 may be callables e -> that expert's
    matrix (to avoid converting every expert); rows are grouped per expert."""
    experts = np.asarray(experts)
    x_rows = _f64(x_rows)
    d = x_rows.shape[1]
    out = np.zeros((len(experts), d))
    get = lambda W, e: W(e) if callable(W) else W[e]
    for e in np.unique(experts):
        sel = np.nonzero(experts == e)[0]
        W1e, W2e = _f64(get(W1, e)), _f64(get(W2, e))
        b1e = None if b1 is None else _f64(get(b1, e))
        b2e = None if b2 is None else _f64(get(b2, e))
        h = W1e.shape[0]
        m = len(sel)
        # Keep every array alive across the call (ctypes holds raw addresses only).
        xs = np.ascontiguousarray(x_rows[sel])
        ids = np.zeros((m, 1), np.int32)
        ones = np.ones((m, 1))
        W1b, W2b = np.ascontiguousarray(W1e[None]), np.ascontiguousarray(W2e[None])
        b1b = None if b1e is None else np.ascontiguousarray(b1e[None])
        b2b = None if b2e is None else np.ascontiguousarray(b2e[None])
        y = np.zeros((m, d))
        rc = _lib_().oracle_experts_combine(m, d, h, 1, 1, _p(xs), _p(ids), _p(ones), _p(W1b),
                                            _p(b1b), _p(W2b), _p(b2b), _p(y))
        if rc:
            raise ValueError("oracle expert evaluation failed")
        out[sel] = y
    return out


def forward(x, Wg, Wn, bg, eps, W1, b1, W2, b2, k: int, groups: int = 0, k_groups: int = 0):
    """The whole layer.  Returns a dict with y, G, idx, importance, cv2, counts, offsets,
    perm, inv_perm (all numpy; floats in float64)."""
    x, Wg, Wn, bg, eps, W1, b1, W2, b2 = map(_f64, (x, Wg, Wn, bg, eps, W1, b1, W2, b2))
    T, d = x.shape
    n, h, _ = W1.shape
    S = T * k
    out = dict(
        y=np.zeros((T, d)), G=np.zeros((T, k)), idx=np.zeros((T, k), np.int32),
        importance=np.zeros(n), counts=np.zeros(n, np.int32), offsets=np.zeros(n + 1, np.int32),
        perm=np.zeros(max(S, 1), np.int32), inv_perm=np.zeros(max(S, 1), np.int32))
    cv2 = ctypes.c_double(0.0)
    rc = _lib_().oracle_forward(
        T, d, h, n, k, groups, k_groups, _p(x), _p(Wg), _p(Wn), _p(bg), _p(eps), _p(W1), _p(b1),
        _p(W2), _p(b2), _p(out["y"]), _p(out["G"]), _p(out["idx"]), _p(out["importance"]),
        ctypes.addressof(cv2), _p(out["counts"]), _p(out["offsets"]), _p(out["perm"]),
        _p(out["inv_perm"]))
    if rc:
        raise ValueError("oracle_forward: bad arguments")
    out["cv2"] = cv2.value
    out["perm"] = out["perm"][:S]
    out["inv_perm"] = out["inv_perm"][:S]
    return out


def backward(x, Wg, Wn, bg, eps, W1, b1, W2, b2, dy, k: int, w_imp: float = 0.0):
    """Gradients of L = sum_t <dy_t, y_t> + w_imp * CV^2(importance) for the
    flat layer, the selection held fixed.  Returns a dict with dx, dWg, dWn,
    dbg, dW1, db1, dW2, db2 (float64, the shapes of the inputs; a bias given as
    None counts as zero and still gets its gradient) and the forward's idx, G."""
    x, Wg, Wn, bg, eps, W1, b1, W2, b2, dy = map(_f64, (x, Wg, Wn, bg, eps, W1, b1, W2, b2, dy))
    T, d = x.shape
    n, h, _ = W1.shape
    out = dict(dx=np.zeros((T, d)), dWg=np.zeros((d, n)), dWn=np.zeros((d, n)), dbg=np.zeros(n),
               dW1=np.zeros((n, h, d)), db1=np.zeros((n, h)), dW2=np.zeros((n, d, h)),
               db2=np.zeros((n, d)), idx=np.zeros((T, k), np.int32), G=np.zeros((T, k)))
    rc = _lib_().oracle_backward_flat(
        T, d, h, n, k, _p(x), _p(Wg), _p(Wn), _p(bg), _p(eps), _p(W1), _p(b1), _p(W2), _p(b2),
        _p(dy), float(w_imp), _p(out["dx"]), _p(out["dWg"]), _p(out["dWn"]), _p(out["dbg"]),
        _p(out["dW1"]), _p(out["db1"]), _p(out["dW2"]), _p(out["db2"]), _p(out["idx"]), _p(out["G"]))
    if rc:
        raise ValueError("oracle_backward_flat: bad arguments")
    return out


def forward_balanced(x, Wg, Wn, bg, eps, thr, W1, b1, W2, b2, k: int):
    """Flat layer with balanced routing: thr None = batchwise mask (every expert
    keeps the floor(k*T/n) tokens with the largest noisy score), else expert e
    keeps the tokens whose score exceeds thr[e].  Returns dict(y [T,d],
    counts [n] int32, W [T,n] the softmax weights over each token's kept
    experts, 0 elsewhere)."""
    x, Wg, Wn, bg, eps, thr, W1, b1, W2, b2 = map(_f64, (x, Wg, Wn, bg, eps, thr, W1, b1, W2, b2))
    T, d = x.shape
    n, h, _ = W1.shape
    out = dict(y=np.zeros((T, d)), counts=np.zeros(n, np.int32), W=np.zeros((T, n)))
    rc = _lib_().oracle_forward_balanced(T, d, h, n, k, _p(x), _p(Wg), _p(Wn), _p(bg), _p(eps),
                                         _p(thr), _p(W1), _p(b1), _p(W2), _p(b2), _p(out["y"]),
                                         _p(out["counts"]), _p(out["W"]))
    if rc:
        raise ValueError("oracle_forward_balanced: bad arguments")
    return out


def ep_regroup(recv_counts):
    """Merged order of the rows one rank receives in the expert-parallel layer
    ("Outrageously Large Neural Networks - 中文验证版", section 方法适配: the
    devices' batches are merged at each expert).  recv_counts [P, nl]: rows of
    local expert e sent by rank q; the received rows come ordered by q, then
    e, then the sender's order.  The merged order puts every expert's rows
    together, rank 0's first: a stable sort of the received rows by expert.
    Returns offsets [nl+1], perm [R] (merged row -> received row), inv [R]."""
    c = np.asarray(recv_counts, dtype=np.int64)
    P, nl = c.shape
    if (c < 0).any():
        raise ValueError("negative count")
    expert_of_row = np.repeat(np.tile(np.arange(nl), P), c.reshape(-1))
    perm = np.argsort(expert_of_row, kind="stable").astype(np.int32)
    offsets = np.concatenate([[0], np.cumsum(c.sum(axis=0))]).astype(np.int32)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size, dtype=np.int32)
    return offsets, perm, inv



def backward_hier(x, Wg, Wn, bg, eps, W1, b1, W2, b2, dy, k: int, groups: int, k_groups: int,
                  w_imp: float = 0.0):
    """Gradients of L = sum_t <dy_t, y_t> + w_imp * CV^2(importance) for the
    hierarchical layer ("MoE:稀疏门控混合专家", section 三: the two-level choice,
    k_groups groups by their noisy score, then k/k_groups experts in each kept
    group by that group's columns; weight = group weight x inner weight), the
    selection held fixed (the oracle's own gate_hier).  Score columns: groups
    0..G-1, then expert e at G + e.  The chain, per token, with c the clean
    score x.Wg + bg and r = x.Wn of a column:
        dG_s   = <dy, E_s> + w_imp dCV^2/dimp_e                   (slot s = (q, j))
        Gp_q   = sum_j G_qj,  Gi_qj = G_qj / Gp_q
        dGp_q  = sum_j dG_qj Gi_qj,  dGi_qj = dG_qj Gp_q
        dHi_qj = Gi_qj (dGi_qj - sum_l Gi_ql dGi_ql)               (inner softmax)
        dHp_q  = Gp_q (dGp_q - sum_l Gp_l dGp_l)                   (group softmax)
        each column's dH gives dc = dH and dr = dH eps sigmoid(r); dx gets
        dc Wg[:, col] + dr Wn[:, col]; dWg[:, col] += dc x, dWn[:, col] += dr x,
        dbg[col] += dc
    and the experts as in `backward`.  Plain numpy in float64; returns the same
    dict as `backward` (dWg, dWn, dbg over all G + n columns)."""
    x, Wg, Wn, bg, eps, W1, b1, W2, b2, dy = map(_f64, (x, Wg, Wn, bg, eps, W1, b1, W2, b2, dy))
    T, d = x.shape
    n, h, _ = W1.shape
    Gn, kg = groups, k_groups
    m, ki = n // Gn, k // kg
    C = Gn + n
    idx, G, _ = gate_hier(x, Wg, Wn, bg, eps, groups, k_groups, k)
    idx = idx.astype(np.int64)
    raw = x @ Wn if (Wn is not None and eps is not None) else None
    # experts: forward pieces per slot, then the chain back
    E = np.zeros((T, k, d))
    dx = np.zeros((T, d))
    dW1, db1 = np.zeros((n, h, d)), np.zeros((n, h))
    dW2, db2 = np.zeros((n, d, h)), np.zeros((n, d))
    for e in range(n):
        tt, jj = np.nonzero(idx == e)
        if tt.size == 0:
            continue
        xs = x[tt]
        z = xs @ W1[e].T + (b1[e] if b1 is not None else 0.0)
        a = np.maximum(z, 0.0)
        E[tt, jj] = a @ W2[e].T + (b2[e] if b2 is not None else 0.0)
        dE = G[tt, jj][:, None] * dy[tt]
        dW2[e] = dE.T @ a
        db2[e] = dE.sum(axis=0)
        dz = (dE @ W2[e]) * (z > 0)
        dW1[e] = dz.T @ xs
        db1[e] = dz.sum(axis=0)
        np.add.at(dx, tt, dz @ W1[e])
    # the importance term, per expert
    imp = np.bincount(idx.ravel(), weights=G.ravel(), minlength=n)
    mu = imp.mean()
    gimp = np.zeros(n)
    if mu != 0.0 and w_imp != 0.0:
        var = ((imp - mu) ** 2).mean()
        gimp = w_imp * (2.0 * (imp - mu) / (n * mu * mu) - 2.0 * var / (n * mu ** 3))
    dG = np.einsum("td,tkd->tk", dy, E) + gimp[idx]
    # two softmax levels
    G3 = G.reshape(T, kg, ki)
    dG3 = dG.reshape(T, kg, ki)
    Gp = G3.sum(axis=2)
    Gi = G3 / Gp[:, :, None]
    dGp = (dG3 * Gi).sum(axis=2)
    dGi = dG3 * Gp[:, :, None]
    dHi = Gi * (dGi - (Gi * dGi).sum(axis=2, keepdims=True))
    dHp = Gp * (dGp - (Gp * dGp).sum(axis=1, keepdims=True))
    # the score columns of every kept (token, column) pair
    cols = np.concatenate([idx[:, ::ki] // m, Gn + idx], axis=1)        # [T, kg + k]
    dH = np.concatenate([dHp, dHi.reshape(T, k)], axis=1)
    dWg, dWn, dbg = np.zeros((d, C)), np.zeros((d, C)), np.zeros(C)
    for q in range(cols.shape[1]):
        c = cols[:, q]
        dc = dH[:, q]
        dx += dc[:, None] * Wg[:, c].T
        np.add.at(dWg.T, c, dc[:, None] * x)
        np.add.at(dbg, c, dc)
        if raw is not None:
            dr = dc * eps[np.arange(T), c] / (1.0 + np.exp(-raw[np.arange(T), c]))
            dx += dr[:, None] * Wn[:, c].T
            np.add.at(dWn.T, c, dr[:, None] * x)
    return dict(dx=dx, dWg=dWg, dWn=dWn, dbg=dbg, dW1=dW1, db1=db1, dW2=dW2, db2=db2,
                idx=idx.astype(np.int32), G=G)
