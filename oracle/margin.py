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


def column_cut_gaps(H: np.ndarray, ranks) -> np.ndarray:
    """For each column e of the oracle scores H [T, n], the gap between its
    ranks[e]-th and (ranks[e]+1)-th largest value (+inf when the rank is 0 or T)."""
    T, n = H.shape
    gaps = np.full(n, np.inf)
    for e in range(n):
        r = int(ranks[e])
        if 0 < r < T:
            part = -np.partition(-H[:, e], (r - 1, r))
            gaps[e] = part[r - 1] - part[r]
    return gaps


def enforce_cut_margin(w: wl.Workload, inp: dict, ranks, min_margin: float = 1e-3,
                       max_redraws: int = 200000) -> int:
    """Balanced routing keeps, in column e, the ranks[e] tokens with the largest
    noisy score H[:, e].  Redraw single eps cells (in place) until every
    column's ranks[e]-th and (ranks[e]+1)-th oracle scores differ by at least
    `min_margin`, so that the kept set has one right answer under rounding.

    Only the cell eps[t, e] of the token t at rank ranks[e] + 1 of a failing
    column is redrawn: that moves H[t, e] alone and leaves every other column
    as it was.  Returns the number of redraws.  Needs noisy flat inputs."""
    if inp["eps"] is None or w.groups:
        raise ValueError("the cut margin redraws eps cells of a flat noisy workload")
    _, _, H, _ = gate_flat(inp["x"], inp["Wg"], inp["Wn"], inp["bg"], inp["eps"], 1)
    T, n = H.shape
    attempts = {}
    redraws = 0
    for e in range(n):
        r = int(ranks[e])
        if not 0 < r < T:
            continue
        while True:
            col = H[:, e]
            order = np.argsort(-col, kind="stable")
            if col[order[r - 1]] - col[order[r]] >= min_margin:
                break
            if redraws >= max_redraws:
                raise RuntimeError(f"column {e}: cut margin not reached after {redraws} redraws")
            t = int(order[r])
            a = attempts.get((t, e), 0) + 1
            attempts[(t, e)] = a
            inp["eps"][t, e] = wl.eps_cell(w, t, e, a)
            # the oracle's noisy score of this one token again (its other columns are unchanged)
            _, _, Ht, _ = gate_flat(inp["x"][t:t + 1], inp["Wg"], inp["Wn"], inp["bg"],
                                    inp["eps"][t:t + 1], 1)
            H[t, e] = Ht[0, e]
            redraws += 1
    return redraws
