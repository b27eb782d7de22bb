"""Test helpers for the expert-parallel layer.

OracleOps: the per-rank steps of ExpertParallelMoE done by the CPU oracle
(fp64), so that the host logic and the exchange run on gloo ranks without a
GPU.  drive_local: runs the phases of P layer objects in one process, with
the all-to-all done by plain tensor copies (no collective); each rank's
kernels are launched one after another and never wait on each other.
"""
from types import SimpleNamespace

import numpy as np
import torch

import oracle


def shape_ns(T, d, h, n, k, groups=0, k_groups=0, dtype="bf16", noisy=True):
    return SimpleNamespace(T=int(T), d=int(d), h=int(h), n=int(n), k=int(k), groups=int(groups),
                           k_groups=int(k_groups), dtype=dtype, noisy=bool(noisy))


class OracleOps:
    def route(self, shape, x, Wg, Wn, bg, eps):
        if shape.groups:
            idx, G, _ = oracle.gate_hier(x, Wg, Wn, bg, eps, shape.groups, shape.k_groups, shape.k)
        else:
            idx, G, _, _ = oracle.gate_flat(x, Wg, Wn, bg, eps, shape.k)
        counts, offsets, perm, inv, imp, _ = oracle.route(idx, G, shape.n)
        t = torch.from_numpy
        return dict(idx=t(idx), G=t(G), counts=t(counts), offsets=t(offsets), perm=t(perm),
                    inv=t(inv), importance=t(imp))

    def gather_rows(self, src, rows, div):
        return src[rows.long() // div].clone()

    def regroup(self, P, n_local, recv_counts, R):
        offsets, perm, inv = oracle.ep_regroup(recv_counts.numpy().reshape(P, n_local))
        assert offsets[-1] == R
        return torch.from_numpy(offsets), torch.from_numpy(perm), torch.from_numpy(inv)

    def experts(self, shape_local, rows, perm, offsets, W1, b1, W2, b2):
        off = offsets.numpy()
        experts = np.repeat(np.arange(off.size - 1), np.diff(off))
        Y = oracle.expert_rows(rows.numpy()[perm.numpy()], experts, W1, b1, W2, b2)
        return torch.from_numpy(Y)

    def combine(self, shape, yslot, inv, G):
        return torch.from_numpy(oracle.combine_rows(yslot.numpy(), inv.numpy(), G.numpy()))

    def cv2(self, importance):
        v = importance.numpy().astype(np.float64)
        m = v.mean()
        return torch.tensor([((v - m) ** 2).mean() / (m * m) if m != 0 else 0.0])


def f64(t):
    return None if t is None else torch.as_tensor(t).double()


def local_experts(inp, first, n_local):
    """This rank's share of the expert weights."""
    sl = slice(first, first + n_local)
    return (inp["W1"][sl], None if inp["b1"] is None else inp["b1"][sl], inp["W2"][sl],
            None if inp["b2"] is None else inp["b2"][sl])


def drive_local(layers, xs, gate, experts):
    """One call of P layers (ranks 0..P-1) in this process.  xs[q]: rank q's
    tokens; gate = (Wg, Wn, bg); eps passed per rank in gate[3][q];
    experts[q] = (W1, b1, W2, b2) of rank q.  Returns per-rank dicts with y,
    idx, G, counts, the merged importance and rows_in."""
    P = len(layers)
    Wg, Wn, bg, epss = gate
    sts = [layers[q].send_phase(xs[q], Wg, Wn, bg, epss[q]) for q in range(P)]
    nl = layers[0].n_local
    # counts all-to-all: rank q receives block q of every rank's counts
    recv_counts = [torch.cat([sts[r]["counts"][q * nl:(q + 1) * nl] for r in range(P)])
                   for q in range(P)]
    # rows all-to-all: rank q receives, from each r in order, r's rows for q
    def block(st, q):
        off = st["offsets"].cpu().numpy()
        return st["xsend"][int(off[q * nl]):int(off[(q + 1) * nl])]
    xrecv = [torch.cat([block(sts[r], q) for r in range(P)]) for q in range(P)]
    ysend = [layers[q].expert_phase(recv_counts[q], xrecv[q], *experts[q]) for q in range(P)]
    # reverse: rank r gets back, from each q in order, its own rows for q
    outs = []
    for r in range(P):
        parts = []
        for q in range(P):
            sizes = [int(sts[s]["counts"][q * nl:(q + 1) * nl].sum()) for s in range(P)]
            start = sum(sizes[:r])
            parts.append(ysend[q][start:start + sizes[r]])
        yslot = torch.cat(parts)
        y = layers[r].combine_phase(sts[r], yslot)
        outs.append(dict(y=y, idx=sts[r]["idx"], G=sts[r]["G"], counts=sts[r]["counts"],
                         rows_in=xrecv[r].shape[0]))
    imp = sum(st["importance"] for st in sts)
    for o in outs:
        o["importance"] = imp
    return outs
