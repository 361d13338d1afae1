"""Flattened-tree structure: depth, position ids, ancestor sets.

Graft page, section 2 (third gear): the hybrid candidate tree is flattened
into one sequence and its tree position encoding and attention mask are
rebuilt before the single verification forward.  SpecOPD page, section 02
(attention-architecture table, full attention row): the mask is the
topological ancestor relation — a node sees its own ancestor path and the
shared trunk, never a sibling branch or a later trunk token.

Readings used here:
  * ``parent`` holds request-local indices, parents precede children, and
    ``-1`` marks a root (one root per request, or one per branch of a
    SpecOPD proposal forest);
  * node i of request r sees the first ``vis[i]`` prefix tokens, where
    ``vis[i] = vis_prefix[i]`` if given, else the whole prefix ``P_r``;
  * the position id of node i is ``vis[i] + depth(i)``: the root sits right
    after the visible prefix.
"""
from __future__ import annotations

import numpy as np


def path_to_root(parent: np.ndarray, n0: int, i: int) -> list[int]:
    """Request-local node indices from the root down to node i (inclusive)."""
    path = []
    j = i
    while j != -1:
        path.append(j)
        j = int(parent[n0 + j])
    path.reverse()
    return path


def tree_prep(parent, node_off, prefix_len, vis_prefix=None, anc_words=None):
    """Per node: depth, position id, visible prefix length and the ancestor
    bitmask (bit j of word j//64 set iff node j is node i or an ancestor).

    Returns (depth int32 [n], pos int32 [n], anc uint64 [n, W], vis int32 [n])."""
    parent = np.asarray(parent)
    node_off = np.asarray(node_off)
    B = node_off.size - 1
    n = int(node_off[-1])
    max_nodes = int(max(node_off[r + 1] - node_off[r] for r in range(B))) if B else 0
    W = anc_words if anc_words is not None else max(1, (max_nodes + 63) // 64)
    depth = np.zeros(n, np.int32)
    pos = np.zeros(n, np.int32)
    vis = np.zeros(n, np.int32)
    anc = np.zeros((n, W), np.uint64)
    for r in range(B):
        n0, n1 = int(node_off[r]), int(node_off[r + 1])
        for i in range(n1 - n0):
            path = path_to_root(parent, n0, i)
            depth[n0 + i] = len(path) - 1
            v = int(prefix_len[r]) if vis_prefix is None else int(vis_prefix[n0 + i])
            vis[n0 + i] = v
            pos[n0 + i] = v + len(path) - 1
            for j in path:
                anc[n0 + i, j // 64] |= np.uint64(1) << np.uint64(j % 64)
    return depth, pos, anc, vis
