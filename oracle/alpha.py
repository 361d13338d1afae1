"""Distribution overlap alpha = 1 - TV(p, q), its prefix product, softmax mass.

SpecOPD page section 03: under exact rejection sampling a drafted token is
accepted with probability equal to the overlap of the draft and target
distributions, i.e. one minus their total-variation distance, and the
expected run of consecutive acceptances along a branch is governed by the
running product of those overlaps (the E2E-TV objective).  Graft page
section 3: the coverage gain of added candidates is the target probability
mass they cover — the softmax mass of given tokens.

Definitions (fp64):
  p = softmax(lp), q = softmax(lq)         per row
  alpha        = sum_v min(p_v, q_v)
  alpha_tv     = 1 - 0.5 * sum_v |p_v - q_v|   (the same number; self-check)
  alpha_prefix = running product of alpha within each branch, in row order
  p_mass       = p[mass_tok]
"""
from __future__ import annotations

import numpy as np

from .attention import as_f64


def softmax(x: np.ndarray) -> np.ndarray:
    m = x.max()
    e = np.exp(x - m)
    return e / e.sum()


def tv_alpha(lp, lq, branch_off=None, mass_tok=None, rows=None):
    """Returns alpha [R], alpha_tv [R], alpha_prefix [R] (or None), p_mass [R] (or None)."""
    lp = np.asarray(lp)
    lq = np.asarray(lq)
    R = lp.shape[0]
    rows = range(R) if rows is None else [int(r) for r in rows]
    alpha = np.full(R, np.nan)
    alpha_tv = np.full(R, np.nan)
    p_mass = None if mass_tok is None else np.full(R, np.nan)
    for r in rows:
        p = softmax(as_f64(lp[r]))
        q = softmax(as_f64(lq[r]))
        alpha[r] = np.minimum(p, q).sum()
        alpha_tv[r] = 1.0 - 0.5 * np.abs(p - q).sum()
        if mass_tok is not None:
            p_mass[r] = p[int(mass_tok[r])]
    prefix = None if branch_off is None else branch_prefix(alpha, branch_off)
    return alpha, alpha_tv, prefix, p_mass


def branch_prefix(alpha, branch_off):
    """Running product of alpha within each branch, in row order (rows
    outside every branch are NaN)."""
    prefix = np.full(len(alpha), np.nan)
    for b in range(len(branch_off) - 1):
        run = 1.0
        for r in range(int(branch_off[b]), int(branch_off[b + 1])):
            run *= alpha[r]
            prefix[r] = run
    return prefix
