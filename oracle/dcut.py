"""D-cut: prefix-product confidence scores and batch-global budget selection.

D-cut page, technical summary section 2 (core mechanism and pipeline):
each candidate position gets a prefix-product score s_{i,k} — the
probability that block i survives to depth k — from the drafter's
confidences; all positions of the batch are flattened and ranked globally;
the top K are kept, which leaves each request a contiguous prefix, and they
are packed into a dense verification batch.  The budget ratio is one of
rho in {0.25, 0.50, 0.75, 1.00}; section 1: a step verifies B x (D+1)
tokens.

Definitions (the scores are *defined* in fp32 so that the selection, an
integer result, is reproducible bit for bit):
  s[r, 0] = 1
  s[r, j] = fp32(s[r, j-1] * c[r, j-1])      j = 1..D, strictly left to right
  K(rho)  = floor(rho * B * (D+1) + 0.5)     (rho as given in fp32, product in fp64)
  keep    = the K positions first in the order (s desc, r asc, j asc)
  keep_len[r] = kept positions of request r (a prefix, since s never grows)
  pack_off    = exclusive prefix sum of keep_len (packed-batch offsets)
  pack_idx    = flat indices r*(D+1)+j of kept positions in (r, j) order
"""
from __future__ import annotations

import math

import numpy as np


def prefix_scores(conf: np.ndarray) -> np.ndarray:
    conf = np.asarray(conf, np.float32)
    B, D = conf.shape
    s = np.ones((B, D + 1), np.float32)
    for j in range(1, D + 1):
        s[:, j] = s[:, j - 1] * conf[:, j - 1]     # float32 * float32 -> float32
    return s


def budget(rho: float, total: int) -> int:
    return int(math.floor(float(np.float32(rho)) * total + 0.5))


def select(conf, rhos):
    """Returns s [B, D+1] f32, keep uint8 [n_rho, B, D+1], keep_len int32 [n_rho, B],
    pack_off int32 [n_rho, B+1], pack_idx int32 [n_rho, B*(D+1)] (-1 padded)."""
    s = prefix_scores(conf)
    B, N = s.shape
    total = B * N
    order = sorted(range(total), key=lambda t: (-float(s[t // N, t % N]), t // N, t % N))
    n_rho = len(rhos)
    keep = np.zeros((n_rho, B, N), np.uint8)
    keep_len = np.zeros((n_rho, B), np.int32)
    pack_off = np.zeros((n_rho, B + 1), np.int32)
    pack_idx = np.full((n_rho, total), -1, np.int32)
    for a, rho in enumerate(rhos):
        K = budget(rho, total)
        for t in order[:K]:
            keep[a, t // N, t % N] = 1
        keep_len[a] = keep[a].sum(axis=1)
        pack_off[a, 1:] = np.cumsum(keep_len[a])
        flat = np.nonzero(keep[a].reshape(-1))[0]
        pack_idx[a, :flat.size] = flat
    return s, keep, keep_len, pack_off, pack_idx


def expected_tokens(s, keep):
    """Expected tokens that one verification step yields at each budget: the
    sum of the kept positions' survival probabilities s (a kept root yields the
    target's own next token, s = 1).  This is the expected-gain side of the
    runtime budget choice (D-cut page, technical summary section 2: expected
    MAT from the confidence estimates), summed over the batch.  Exact sum
    (math.fsum of the fp32 scores), returned as float64 [n_rho]."""
    s = np.asarray(s, np.float32)
    return np.array([math.fsum(float(x) for x in s[keep[a].astype(bool)]) for a in range(keep.shape[0])],
                    np.float64)


def choose_rho(E, cost):
    """rho* index = argmax over budgets of E[a] / cost[a], the expected gain
    over the profiled step cost (same section: the ratio of expected MAT to
    the hardware-profiled run cost); the lowest index on ties.  The cost table
    is an input (its calibration is out of scope)."""
    best, arg = -math.inf, -1
    for a in range(len(E)):
        v = float(E[a]) / float(cost[a])
        if v > best:
            best, arg = v, a
    return arg
