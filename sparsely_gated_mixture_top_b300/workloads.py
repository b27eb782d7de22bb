"""Synthetic workloads of the MoE layer forward pass and their seeded inputs.

Each workload fixes the layer's shape and how its inputs are drawn; `make_inputs`
turns it into host tensors with the counter-based generator of `synth`.  The
shapes follow the pages: experts are 512 -> 1024 -> 512 feed-forward nets
("MoE:稀疏门控混合专家", section 二), k = 4 or 2 experts per token
("Outrageously Large Neural Networks - 中文验证版", section 方法适配) and the
hierarchical layer splits 4096 experts into 16 groups of 256, keeping 2 groups
and 2 experts in each ("MoE:稀疏门控混合专家", section 三).  The pages' own
data sets are not available; these synthetic tensors stand in for them.

Distributions: x ~ N(0,1); W_g, W_noise ~ N(0, 1/d); W1 ~ N(0, 2/d);
W2 ~ N(0, 1/h); eps ~ N(0,1); expert biases 0 unless `bias_std` is given.
The skewed workload adds a per-expert bias b_i = 2 log(1/(i+1)) to the clean
gate score, which makes the expert load Zipf-like.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

from . import synth

# Tensor ids of the generator streams (part of the input definition).
TID_X, TID_WG, TID_WN, TID_EPS, TID_W1, TID_B1, TID_W2, TID_B2 = 1, 2, 3, 5, 6, 7, 8, 9
TID_EPS_CELL = 10   # single eps cells redrawn one at a time (attempt >= 1)


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    h: int
    n: int
    k: int
    groups: int = 0          # 0: flat gating; G > 0: hierarchical, G groups of n/G experts
    k_groups: int = 0        # hierarchical: groups kept per token
    dtype: str = "bf16"      # storage type of x, W1, W2, Y and y: "bf16" or "f32"
    noisy: bool = True
    gate_bias: str = "none"  # "none" or "zipf"
    seed: int = 20250
    bias_std: float = 0.0    # expert biases b1, b2 ~ N(0, bias_std^2); 0 means zeros

    @property
    def cols(self) -> int:
        """Gate score columns: n (flat) or G + n (hierarchical)."""
        return self.n if self.groups == 0 else self.groups + self.n

    @property
    def slots(self) -> int:
        return self.T * self.k

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_flat_fp32", T=256, d=512, h=1024, n=8, k=2, dtype="f32", seed=20250),
        Workload("flat_n256_k4", T=16384, d=512, h=1024, n=256, k=4, seed=20251),
        Workload("hier_4096h_16x256", T=32768, d=512, h=1024, n=4096, k=4, groups=16,
                 k_groups=2, seed=20252),
        Workload("skewed_zipf_n64", T=65536, d=1024, h=4096, n=64, k=2, gate_bias="zipf",
                 seed=20253),
        Workload("sparse_n2048_T4096", T=4096, d=512, h=1024, n=2048, k=4, seed=20254),
        Workload("sparse_n2048_T32768", T=32768, d=512, h=1024, n=2048, k=4, seed=20254),
        Workload("sparse_n2048_T131072", T=131072, d=512, h=1024, n=2048, k=4, seed=20254),
    ]
}


def _torch_dtype(dt: str):
    return {"bf16": torch.bfloat16, "f32": torch.float32}[dt]


def normal_tensor(w: Workload, tid: int, shape, scale: float, dtype: str, attempt: int = 0,
                  start: int = 0, pin: bool = False) -> torch.Tensor:
    """Elements [start, start + numel) of generator stream `tid`, scaled, as a tensor."""
    count = 1
    for s in shape:
        count *= int(s)
    out = torch.empty(tuple(shape), dtype=_torch_dtype(dtype), pin_memory=pin)
    if count:
        synth.fill_normal(out, w.seed, tid, attempt, start, scale)
    return out


def gate_bias(w: Workload) -> torch.Tensor | None:
    if w.gate_bias == "none":
        return None
    if w.gate_bias == "zipf":
        b = torch.zeros(w.cols, dtype=torch.float32)
        off = 0 if w.groups == 0 else w.groups
        b[off:off + w.n] = torch.tensor([2.0 * math.log(1.0 / (i + 1)) for i in range(w.n)],
                                        dtype=torch.float64).float()
        return b
    raise ValueError(f"unknown gate bias {w.gate_bias!r}")


def expert_weight(w: Workload, which: str, e: int) -> torch.Tensor:
    """W1[e] ([h, d]) or W2[e] ([d, h]) alone, identical to the slice of the full tensor."""
    if which == "W1":
        return normal_tensor(w, TID_W1, (w.h, w.d), math.sqrt(2.0 / w.d), w.dtype,
                             start=e * w.h * w.d)
    if which == "W2":
        return normal_tensor(w, TID_W2, (w.d, w.h), math.sqrt(1.0 / w.h), w.dtype,
                             start=e * w.d * w.h)
    raise ValueError(which)


def expert_bias(w: Workload, which: str, e: int) -> torch.Tensor:
    size = w.h if which == "b1" else w.d
    if w.bias_std == 0.0:
        return torch.zeros(size, dtype=torch.float32)
    tid = TID_B1 if which == "b1" else TID_B2
    return normal_tensor(w, tid, (size,), w.bias_std, "f32", start=e * size)


def eps_rows(w: Workload, rows, attempts) -> torch.Tensor:
    """eps rows for the given tokens, each drawn with its own attempt counter."""
    out = torch.empty((len(rows), w.cols), dtype=torch.float32)
    for i, (t, a) in enumerate(zip(rows, attempts)):
        synth.fill_normal(out[i], w.seed, TID_EPS, int(a), int(t) * w.cols, 1.0)
    return out


def eps_cell(w: Workload, t: int, e: int, attempt: int) -> float:
    """A fresh N(0,1) draw for the single cell eps[t, e] (stream TID_EPS_CELL,
    its own attempt counter), for redraws that must move one score only."""
    out = torch.empty((1,), dtype=torch.float32)
    synth.fill_normal(out, w.seed, TID_EPS_CELL, int(attempt), int(t) * w.cols + int(e), 1.0)
    return float(out[0])


def make_inputs(w: Workload, pin: bool = False, experts: bool = True,
                tokens: slice | None = None) -> dict:
    """All inputs of the layer as host tensors.

    x [T,d]; Wg, Wn [d,C] fp32; bg [C] fp32 or None; eps [T,C] fp32 or None;
    W1 [n,h,d]; b1 [n,h] fp32; W2 [n,d,h]; b2 [n,d] fp32 (W1/W2/x in w.dtype).
    `experts=False` skips the expert weights; `tokens` restricts x/eps to a
    range of token rows (their values equal the same rows of the full tensors).
    """
    t0, t1 = (0, w.T) if tokens is None else (tokens.start or 0, tokens.stop)
    nt = t1 - t0
    C = w.cols
    inp = {
        "x": normal_tensor(w, TID_X, (nt, w.d), 1.0, w.dtype, start=t0 * w.d, pin=pin),
        "Wg": normal_tensor(w, TID_WG, (w.d, C), math.sqrt(1.0 / w.d), "f32", pin=pin),
        "Wn": normal_tensor(w, TID_WN, (w.d, C), math.sqrt(1.0 / w.d), "f32", pin=pin),
        "bg": gate_bias(w),
        "eps": (normal_tensor(w, TID_EPS, (nt, C), 1.0, "f32", start=t0 * C, pin=pin)
                if w.noisy else None),
    }
    if experts:
        inp["W1"] = normal_tensor(w, TID_W1, (w.n, w.h, w.d), math.sqrt(2.0 / w.d), w.dtype,
                                  pin=pin)
        inp["W2"] = normal_tensor(w, TID_W2, (w.n, w.d, w.h), math.sqrt(1.0 / w.h), w.dtype,
                                  pin=pin)
        if w.bias_std == 0.0:
            inp["b1"] = torch.zeros((w.n, w.h), dtype=torch.float32)
            inp["b2"] = torch.zeros((w.n, w.d), dtype=torch.float32)
        else:
            inp["b1"] = normal_tensor(w, TID_B1, (w.n, w.h), w.bias_std, "f32")
            inp["b2"] = normal_tensor(w, TID_B2, (w.n, w.d), w.bias_std, "f32")
    return inp
