"""Per-row reductions over the target's next-token logits (fp64).

Graft page section 2 (second and third gears): each table row stores the
top-k most probable next tokens, ranked by probability, and every verified
position's next-token distribution updates the row of its token; the
verification accepts a draft token only when it is what the target model
picks (greedy verification: the argmax).  Section 5 puts the useful width
at about 8.

Definitions:
  * argmax  = the smallest index attaining the row maximum;
  * top-k   = the first k entries of the row ordered by (value descending,
              index ascending);
  * row_max = the maximum value;
  * row_lse = row_max + log(sum(exp(x - row_max))), natural log.
Ranking by logit equals ranking by probability (softmax is monotone).
"""
from __future__ import annotations

import numpy as np

from .attention import as_f64


def topk_row(x: np.ndarray, k: int) -> np.ndarray:
    """Indices of the top-k of one row under (value desc, index asc).

    Exact: every member of the top-k is >= the k-th largest value, so the
    candidates ``x >= kth`` (ascending index) contain it; a stable sort of
    the candidates by descending value keeps equal values in index order."""
    V = x.size
    kth = np.partition(x, V - k)[V - k]
    cand = np.nonzero(x >= kth)[0]
    order = np.argsort(-x[cand], kind="stable")
    return cand[order[:k]]


def argmax_topk(logits, k: int, rows=None):
    """Returns argmax int32 [R], topk_idx int32 [R, k], topk_val float32 [R, k],
    row_max float32 [R], row_lse float64 [R] for the given rows (all by default)."""
    x_all = np.asarray(logits)
    rows = range(x_all.shape[0]) if rows is None else [int(r) for r in rows]
    R = len(rows)
    argmax = np.empty(R, np.int32)
    tk_idx = np.empty((R, k), np.int32)
    tk_val = np.empty((R, k), np.float32)
    rmax = np.empty(R, np.float32)
    rlse = np.empty(R, np.float64)
    for t, r in enumerate(rows):
        x = as_f64(x_all[r])
        m = x.max()
        argmax[t] = int(np.nonzero(x == m)[0][0])
        if k > 0:
            idx = topk_row(x, k)
            tk_idx[t] = idx
            tk_val[t] = x[idx]
        rmax[t] = m
        rlse[t] = m + np.log(np.exp(x - m).sum())
    return argmax, tk_idx, tk_val, rmax, rlse
