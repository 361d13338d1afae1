"""Lossless T = 1 verification of a draft tree by rejection sampling.

SpecOPD page §03: under exact rejection sampling the probability that the
target accepts a draft token is the overlap of the draft and target
distributions (alpha = sum min(p, q)); D-cut page §4 and SpecOPD page §04
report temperature-1 results.  The pages give no tree procedure, so this is
the standard multi-candidate scheme (reading, stated here in full):

  start at the root; p' = softmax(target logits at the current node)
  for each child c of the current node, in node-index order, token x:
      q = softmax(draft logits at the current node)   (c was drawn from q)
      accept c  iff  u[c] < min(1, p'(x) / q(x))      (u: an input uniform)
      on acceptance: the current node becomes c, p' = softmax(target at c),
                     and its children are tried next
      on rejection:  p' = max(0, p' - q) / sum max(0, p' - q)   (residual)
  when no child is accepted (or the node has none): the bonus token is drawn
  from p' by inverse CDF in token order: the smallest j with
  sum_{v <= j} p'(v) > u_final.

Each accepted step leaves the emitted token distributed exactly as the
target's next-token distribution, which is what makes the scheme lossless;
the tests pin that property by Monte Carlo.  Arithmetic: float64 from the
logits (bf16 logits are exact in float64).  A residual that sums to 0 (only
possible through rounding: a rejection needs p'(x) < q(x), which leaves
mass where p' > q) restores p' = softmax(target at the current node).
"""
from __future__ import annotations

import numpy as np


def _softmax64(logits):
    x = np.asarray(logits, np.float64)
    m = x.max()
    e = np.exp(x - m)
    return e / e.sum()


def _row(logits, i):
    x = logits[i]
    if x.dtype == np.uint16:          # bf16 bit patterns
        x = (x.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return x


def rejection_verify(parent, tok, p_logits, q_logits, node_off, u_node, u_final, max_depth):
    """Returns accept_len int32 [B] (accepted draft nodes), best_node int32 [B]
    (request-local final node), path int32 [B, max_depth+1] (-1 padded),
    bonus int32 [B], the trace list of (request, node, p_accept) per child
    test, and the distribution each bonus token was drawn from (float64 [V]
    per request) — the last two for test construction."""
    B = len(node_off) - 1
    acc = np.zeros(B, np.int32)
    best = np.zeros(B, np.int32)
    path = np.full((B, max_depth + 1), -1, np.int32)
    bonus = np.zeros(B, np.int32)
    trace = []
    finals = []
    for r in range(B):
        a, b = int(node_off[r]), int(node_off[r + 1])
        n = b - a
        children = [[] for _ in range(n)]
        for i in range(1, n):
            children[int(parent[a + i])].append(i)
        cur, depth = 0, 0
        path[r, 0] = 0
        while True:
            pp = _softmax64(_row(p_logits, a + cur))
            q = _softmax64(_row(q_logits, a + cur))
            nxt = -1
            for c in children[cur]:
                x = int(tok[a + c])
                ratio = 1.0 if q[x] <= 0 else min(1.0, pp[x] / q[x])
                trace.append((r, c, ratio))
                if u_node[a + c] < ratio:
                    nxt = c
                    break
                res = np.maximum(0.0, pp - q)
                z = res.sum()
                pp = res / z if z > 0 else _softmax64(_row(p_logits, a + cur))
            if nxt < 0:
                finals.append(pp)
                cdf = np.cumsum(pp)
                j = int(np.searchsorted(cdf, u_final[r], side="right"))
                bonus[r] = min(j, len(pp) - 1)
                break
            cur = nxt
            depth += 1
            if depth <= max_depth:
                path[r, depth] = cur
        acc[r] = depth
        best[r] = cur
    return acc, best, path, bonus, trace, finals
