"""Host-side data for Graft retrieval: stage templates and hybrid-tree layout.

Graft page §2 (second gear): retrieval expands a subtree from the current
token along a fixed, asymmetric stage-adaptive template — the top-ranked
successor gets more children and a deeper greedy chain, lower ranks fewer —
and the number of retrieval slots is 52, 36, 20 or 0 for the pruning stages
root, depth 1, depth 5 and none (a 60-slot budget).  §5: best depth and width
about 8.

The template is *data* for ``graft_retrieve``: every rank path
(r_1..r_d), d <= depth, r < width, is weighted prod_j 0.9 * 0.4**r_j; the S
heaviest paths form the stage's template, ties going to the
lexicographically smaller path.  A path always weighs less than its prefix,
so the set is prefix-closed and is listed so that parents come first.
Weights are compared exactly as integers: w(d, R) = 9^d 2^R / (10^d 5^R)
for a path of length d with rank sum R.
"""
from __future__ import annotations

import numpy as np

STAGE_SLOTS = (52, 36, 20, 0)      # retrieval slots: pruned at root, depth 1, depth 5, none
STAGE_DRAFT = (8, 24, 40, 60)      # draft nodes kept in the same stages


def _heavier(a, b) -> bool:
    """Path a = (len, rank_sum, ranks) strictly before path b in template order."""
    (da, ra, pa), (db, rb, pb) = a, b
    lhs = 9 ** da * 2 ** ra * 10 ** db * 5 ** rb
    rhs = 9 ** db * 2 ** rb * 10 ** da * 5 ** ra
    if lhs != rhs:
        return lhs > rhs
    return pa < pb


def stage_template(S: int, width: int = 8, depth: int = 8):
    """(tparent, trank) int32 [S] for one stage."""
    chosen: list[tuple] = []
    index: dict[tuple, int] = {}
    frontier = [(1, r, (r,)) for r in range(width)]
    while frontier and len(chosen) < S:
        best = 0
        for i in range(1, len(frontier)):
            if _heavier(frontier[i], frontier[best]):
                best = i
        node = frontier.pop(best)
        index[node[2]] = len(chosen)
        chosen.append(node)
        d, rsum, path = node
        if d < depth:
            frontier.extend((d + 1, rsum + r, path + (r,)) for r in range(width))
    tparent = np.array([index[p[:-1]] if len(p) > 1 else -1 for _, _, p in chosen], np.int32)
    trank = np.array([p[-1] for _, _, p in chosen], np.int32)
    return tparent, trank


def stage_templates(width: int = 8, depth: int = 8, slots=STAGE_SLOTS):
    """All stages concatenated: tparent, trank int32 [sum S], tmpl_off int32 [n_stage + 1]."""
    parts = [stage_template(S, width, depth) for S in slots]
    off = np.concatenate([[0], np.cumsum([len(p[0]) for p in parts])]).astype(np.int32)
    tp = np.concatenate([p[0] for p in parts]).astype(np.int32)
    tr = np.concatenate([p[1] for p in parts]).astype(np.int32)
    return tp, tr, off


def assemble_hybrid(parent_draft: np.ndarray, tparent_stage: np.ndarray) -> np.ndarray:
    """Parent array of the hybrid tree: the draft tree (root = node 0) followed
    by the retrieval slots, whose template roots hang off the tree root."""
    nd = parent_draft.size
    rp = np.where(tparent_stage < 0, 0, tparent_stage + nd).astype(np.int32)
    return np.concatenate([parent_draft.astype(np.int32), rp])
