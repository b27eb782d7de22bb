"""Top-k margin enforcement for synthetic inputs (test infrastructure only).

A token whose k-th and (k+1)-th noisy scores differ by less than `min_margin`
(at either level of a hierarchical gate) has more than one top-k set that
rounding could produce.  Such a token gets its eps row redrawn from the
generator with the next attempt counter, and only that token's gate is
recomputed, until every checked token clears the margin.
"""
from __future__ import annotations

import numpy as np

from sparsely_gated_mixture_top_b300 import workloads as wl

from . import gate_flat, gate_hier


def gate_margins(w: wl.Workload, inp: dict, rows) -> np.ndarray:
    """Oracle top-k margin of the given token rows."""
    rows = np.asarray(rows, dtype=np.int64)
    x = inp["x"][rows]
    eps = None if inp["eps"] is None else inp["eps"][rows]
    if w.groups == 0:
        _, _, _, margin = gate_flat(x, inp["Wg"], inp["Wn"], inp["bg"], eps, w.k)
    else:
        _, _, margin = gate_hier(x, inp["Wg"], inp["Wn"], inp["bg"], eps, w.groups, w.k_groups,
                                 w.k)
    return margin


def enforce_margin(w: wl.Workload, inp: dict, rows=None, min_margin: float = 1e-3,
                   max_rounds: int = 64) -> int:
    """Redraw eps rows (in place, in inp["eps"]) until every row in `rows` (default:
    all tokens) has an oracle top-k margin >= min_margin.  Returns the number of
    redraws.  Needs noisy inputs (an eps tensor)."""
    if inp["eps"] is None:
        raise ValueError("margin enforcement redraws eps; the workload has no noise")
    rows = np.arange(inp["x"].shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    attempts = {}
    todo = rows
    redraws = 0
    for _ in range(max_rounds):
        margin = gate_margins(w, inp, todo)
        todo = todo[margin < min_margin]
        if todo.size == 0:
            return redraws
        for t in todo.tolist():
            attempts[t] = attempts.get(t, 0) + 1
        inp["eps"][todo] = wl.eps_rows(w, todo.tolist(), [attempts[t] for t in todo.tolist()])
        redraws += int(todo.size)
    raise RuntimeError(f"{todo.size} tokens still below the margin after {max_rounds} rounds")
