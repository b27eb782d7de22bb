"""Expert-parallel MoE layer over a torch.distributed process group.

The pages' own system keeps the experts on different devices and moves each
token's rows to its experts and back by all-to-all ("Outrageously Large
Neural Networks - MoE 怎样让模型'很大但不每次全算'", section 方法怎么做);
each device holds a share of the experts and the devices' batches are merged
at the MoE layer, so that each expert runs once on the rows of every device
("Outrageously Large Neural Networks - 中文验证版", sections 计算设置 and
方法适配).

Partition: P ranks, n % P == 0; rank q owns experts [q*n/P, (q+1)*n/P).  Each
rank gates its own tokens against all n experts (the gate matrices are
replicated), so the rows bound for rank q are one contiguous range of its
dispatch order.  The sequence of one call is the one include/moe_ep.h lists:
local gate + dispatch, row pack, counts and rows all-to-all, regroup into the
merged expert order, the local experts, rows back by the reverse
all-to-all, combine; the importance vector is summed over the ranks and its
CV^2 taken on the merged batch.

Every arithmetic step runs in libmoe_b300.so (`CudaOps`); this module only
sizes buffers, computes the split sizes on the host (one copy of 2n int32
per call) and calls the collectives (NCCL on GPUs).  `ops` is a parameter so
that the host logic and the exchange can be exercised on CPU ranks (gloo)
with another implementation of the same per-rank steps.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist


class CudaOps:
    """The per-rank steps on one GPU, through the C ABI."""

    def __init__(self, device=None):
        from . import binding as B
        self.B = B
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None \
            else torch.device(device)
        self._ws = {}

    def _workspace(self, key, shape):
        need = self.B.workspace_bytes(shape)
        ws = self._ws.get(key)
        if ws is None or ws.numel() < need:
            ws = self.B.workspace(shape, self.device)
            self._ws[key] = ws
        return ws

    def route(self, shape, x, Wg, Wn, bg, eps):
        B = self.B
        ws = self._workspace("layer", shape)
        T, k, n = shape.T, shape.k, shape.n
        dev = self.device
        idx = torch.empty((T, k), dtype=torch.int32, device=dev)
        G = torch.empty((T, k), dtype=torch.float32, device=dev)
        counts = torch.empty(n, dtype=torch.int32, device=dev)
        offsets = torch.empty(n + 1, dtype=torch.int32, device=dev)
        perm = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
        inv = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
        imp = torch.empty(n, dtype=torch.float32, device=dev)
        cv2 = torch.empty(1, dtype=torch.float32, device=dev)
        if T > 0:
            B.moe_gate(shape, x, Wg, Wn, bg, eps, idx, G, ws)
        B.moe_dispatch(shape, idx, G, counts, offsets, perm, inv, imp, cv2, ws)
        return dict(idx=idx, G=G, counts=counts, offsets=offsets, perm=perm[:T * k],
                    inv=inv[:T * k], importance=imp)

    def gather_rows(self, src, rows, div):
        dst = torch.empty((rows.numel(), src.shape[1]), dtype=src.dtype, device=src.device)
        self.B.moe_gather_rows(src, rows, div, dst, self._ws.get("layer"))
        return dst

    def regroup(self, P, n_local, recv_counts, R):
        dev = self.device
        offsets = torch.empty(n_local + 1, dtype=torch.int32, device=dev)
        perm = torch.empty(max(R, 1), dtype=torch.int32, device=dev)
        inv = torch.empty(max(R, 1), dtype=torch.int32, device=dev)
        self.B.moe_ep_regroup(P, n_local, recv_counts, R, offsets, perm, inv,
                              self._ws.get("layer"))
        return offsets, perm[:R], inv[:R]

    def experts(self, shape_local, rows, perm, offsets, W1, b1, W2, b2):
        ws = self._workspace("experts", shape_local)
        Y = torch.empty((shape_local.T, shape_local.d), dtype=rows.dtype, device=rows.device)
        self.B.moe_expert_ffn(shape_local, rows, perm, offsets, W1, b1, W2, b2, Y, ws)
        return Y

    def combine(self, shape, yslot, inv, G):
        y = torch.empty((shape.T, shape.d), dtype=yslot.dtype, device=yslot.device)
        self.B.moe_combine(shape, yslot, inv, G, y, self._ws["layer"])
        return y

    def cv2(self, importance):
        out = torch.empty(1, dtype=torch.float32, device=importance.device)
        self.B.moe_importance_cv2(importance, out)
        return out

    def check(self):
        for ws in self._ws.values():
            status = self.B.moe_check(ws)
            if status != self.B.MOE_OK:
                raise self.B.MoEError("expert-parallel layer", status)


def split_sizes(counts: np.ndarray, recv_counts: np.ndarray, P: int) -> tuple[list, list]:
    """Rows this rank sends to and receives from each rank: the sums of its
    own counts over each rank's expert block, and of the counts it received."""
    nl = counts.size // P
    send = counts.reshape(P, nl).sum(axis=1)
    recv = recv_counts.reshape(P, nl).sum(axis=1)
    return [int(v) for v in send], [int(v) for v in recv]


class ExpertParallelMoE:
    """One MoE layer whose n experts are split over the ranks of `group`.

    shape_fields: dict with d, h, n, k, groups, k_groups, dtype, noisy (the
    token count comes from each call's x).  `make_shape(T, d, h, n, k, ...)`
    builds the per-call ABI shape (binding.make_shape for CudaOps)."""

    def __init__(self, shape_fields: dict, make_shape, group=None, ops=None, ranks=None):
        """ranks = (P, rank) places the layer without a process group (its
        phases are then driven by the caller; `forward` needs the group)."""
        self.f = dict(shape_fields)
        self.make_shape = make_shape
        self.group = group
        if ranks is None:
            self.P, self.rank = dist.get_world_size(group), dist.get_rank(group)
        else:
            self.P, self.rank = int(ranks[0]), int(ranks[1])
        n = self.f["n"]
        if n % self.P:
            raise ValueError(f"n = {n} experts do not split over {self.P} ranks")
        self.n_local = n // self.P
        self.first_expert = self.rank * self.n_local
        self.ops = CudaOps() if ops is None else ops

    def _shape(self, T, n=None, k=None, groups=None, k_groups=None, noisy=None):
        f = self.f
        return self.make_shape(T, f["d"], f["h"], f["n"] if n is None else n,
                               f["k"] if k is None else k,
                               f.get("groups", 0) if groups is None else groups,
                               f.get("k_groups", 0) if k_groups is None else k_groups,
                               f["dtype"], f.get("noisy", True) if noisy is None else noisy)

    # The three local phases of a call; `forward` runs them around the
    # collectives.  Each phase only enqueues this rank's own kernels, so the
    # phases of several ranks can also be driven from one process.
    def send_phase(self, x, Wg, Wn, bg, eps) -> dict:
        """Gate and dispatch this rank's tokens; the send buffer in expert order."""
        shape = self._shape(x.shape[0])
        st = self.ops.route(shape, x, Wg, Wn, bg, eps)
        st["shape"] = shape
        st["xsend"] = self.ops.gather_rows(x, st["perm"], self.f["k"])
        return st

    def expert_phase(self, recv_counts, xrecv, W1, b1, W2, b2):
        """This rank's experts on the merged rows (received order in and out)."""
        R = xrecv.shape[0]
        offsets_l, perm_l, inv_l = self.ops.regroup(self.P, self.n_local, recv_counts, R)
        if R == 0:
            return xrecv
        shape_l = self._shape(R, n=self.n_local, k=1, groups=0, k_groups=0, noisy=False)
        Y = self.ops.experts(shape_l, xrecv, perm_l, offsets_l, W1, b1, W2, b2)
        return self.ops.gather_rows(Y, inv_l, 1)

    def combine_phase(self, st, yslot):
        """y of this rank's tokens from its slot rows (its own expert order)."""
        return self.ops.combine(st["shape"], yslot, st["inv"], st["G"])

    def forward(self, x, Wg, Wn, bg, eps, W1, b1, W2, b2) -> dict:
        """x [T_r, d] this rank's tokens; Wg, Wn, bg the replicated gate;
        W1 [n_local, h, d], b1, W2 [n_local, d, h], b2 this rank's experts.
        Returns y [T_r, d], idx, G, importance and cv2 of the merged batch,
        and rows_in (rows this rank's experts ran on)."""
        grp = self.group
        st = self.send_phase(x, Wg, Wn, bg, eps)
        recv_counts = torch.empty_like(st["counts"])
        dist.all_to_all_single(recv_counts, st["counts"], group=grp)
        send_rows, recv_rows = split_sizes(st["counts"].cpu().numpy(),
                                           recv_counts.cpu().numpy(), self.P)
        xsend = st["xsend"]
        xrecv = xsend.new_empty((sum(recv_rows), xsend.shape[1]))
        dist.all_to_all_single(xrecv, xsend, recv_rows, send_rows, group=grp)
        ysend = self.expert_phase(recv_counts, xrecv, W1, b1, W2, b2)
        yslot = xsend.new_empty(xsend.shape)
        dist.all_to_all_single(yslot, ysend, send_rows, recv_rows, group=grp)
        y = self.combine_phase(st, yslot)
        importance = st["importance"].clone()
        dist.all_reduce(importance, group=grp)
        return dict(y=y, idx=st["idx"], G=st["G"], importance=importance,
                    cv2=self.ops.cv2(importance), counts=st["counts"], rows_in=xrecv.shape[0])
