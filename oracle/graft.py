"""Graft's successor table: online update, stage templates, retrieval.

Graft page section 2 (second gear): a V x k integer table lives in GPU
memory; row t holds the k most probable tokens to follow token t.  Retrieval
expands a subtree rooted at the current token by following a fixed
stage-adaptive template over the table; the template is asymmetric — the
top-ranked successor gets more children and a deeper greedy chain, lower
ranks fewer.  The verification budget is 60 slots, split between kept draft
nodes and retrieved nodes as 8/52 (pruned at the root), 24/36 (depth 1),
40/20 (depth 5) and 60/0 (not pruned).  Section 5: the best retrieval depth
and width are both about 8.  Section 2 (third gear) and section 6: after
verification every verified position — accepted or rejected — rewrites the
row of its token with the target's top-k next tokens.

Readings used here:
  * conflicts: when several verified nodes carry the same token, the last in
    (request, node) order wins; the row is overwritten, not merged;
  * template: best-first over rank paths (r_1..r_d), d <= 8, r < k, with
    weight prod_j w(r_j), w(r) = 0.9 * 0.4**r; equal weights are broken by
    the lexicographically smaller path; the first S paths form the template.
    Every path's weight is below its prefix's, so the template is
    prefix-closed and parents precede children.  The pages fix only the
    qualitative shape, so the exact slots are *parity unpinned* against the
    pages (the retrieval given a template is pinned).
  * the retrieved subtree hangs off the tree root (the current token).

Next rows built on the same table (readings, the pages give no procedure):
  * stage decision (section 2, first gear): draft layer L of a node is its
    depth - 1 (the root is the current token, depth 0); its cumulative
    confidence is the fp32 product of the drafter confidences on its path,
    root excluded, in root-to-node order.  At the checkpoints, layers 0, 1
    and 5, the best (largest) cumulative confidence of the layer is compared
    with that checkpoint's calibrated threshold; the first checkpoint below
    its threshold gives the stage 0, 1, 2 (8/52, 24/36, 40/20), none gives 3
    (60/0).  A layer the draft does not reach counts as best = 0.
  * batched static-tree replacement (section 4, batched serving): the
    per-request slot count S stays fixed; draft nodes whose cumulative
    confidence is below the threshold, and their descendants, are replaced
    by retrieval nodes: the first S - kept slots of the best-first template,
    rooted at the current token.  Kept nodes keep their order.
  * Graft-TAIL (section 7): a block draft is a chain; its confident prefix
    (cumulative confidence >= threshold) is kept and the tail is replaced by
    the first retrieval slots of the best-first template, continuing from the
    last kept token (the deepest kept node).
"""
from __future__ import annotations

import heapq
from fractions import Fraction

import numpy as np

STAGE_SLOTS = (52, 36, 20, 0)   # retrieval slots for stages root, depth1, depth5, none


def adj_update(adj, tok, topk_idx, valid=None):
    """In place: for each valid node in order, adj[tok[i], :] = topk_idx[i, :k]."""
    k = adj.shape[1]
    for i in range(len(tok)):
        if valid is not None and not valid[i]:
            continue
        adj[int(tok[i]), :] = topk_idx[i, :k]
    return adj


def stage_template(S, k=8, max_depth=8, w0=Fraction(9, 10), decay=Fraction(2, 5)):
    """First S rank paths in best-first order; returns (tparent, trank) int32 [S].

    tparent[s] is the slot index of the path's prefix (-1 = the root token),
    trank[s] the last rank of the path.  Exact rational weights."""
    w = [w0 * decay ** r for r in range(k)]
    heap = [(-w[r], (r,)) for r in range(k)]
    heapq.heapify(heap)
    slot_of = {}
    tparent, trank = [], []
    while heap and len(tparent) < S:
        negw, path = heapq.heappop(heap)
        slot_of[path] = len(tparent)
        tparent.append(slot_of[path[:-1]] if len(path) > 1 else -1)
        trank.append(path[-1])
        if len(path) < max_depth:
            for r in range(k):
                heapq.heappush(heap, (negw * w[r], path + (r,)))
    return np.array(tparent, np.int32), np.array(trank, np.int32)


def stage_templates(k=8, max_depth=8, slots=STAGE_SLOTS):
    """Concatenated per-stage templates plus offsets [n_stage + 1]."""
    tp, tr, off = [], [], [0]
    for S in slots:
        p, r = stage_template(S, k, max_depth)
        tp.append(p)
        tr.append(r)
        off.append(off[-1] + S)
    return (np.concatenate(tp).astype(np.int32), np.concatenate(tr).astype(np.int32),
            np.array(off, np.int32))


def retrieve(adj, root_tok, stage, tparent, trank, tmpl_off, max_slots):
    """Template expansion per request.  Slot s of request b:
    tok = adj[tok_of(tparent[s]), trank[s]], tok_of(-1) = root_tok[b].
    Returns rtok [B, max_slots], rparent [B, max_slots] (-1 padded) and nslots [B]."""
    B = len(root_tok)
    rtok = np.full((B, max_slots), -1, np.int32)
    rpar = np.full((B, max_slots), -1, np.int32)
    nslots = np.zeros(B, np.int32)
    for b in range(B):
        st = int(stage[b])
        s0, s1 = int(tmpl_off[st]), int(tmpl_off[st + 1])
        for s in range(s1 - s0):
            p = int(tparent[s0 + s])
            src = int(root_tok[b]) if p < 0 else int(rtok[b, p])
            rtok[b, s] = adj[src, int(trank[s0 + s])]
            rpar[b, s] = p
        nslots[b] = s1 - s0
    return rtok, rpar, nslots


def assemble_hybrid(parent_draft, tparent_stage):
    """Hybrid tree = kept draft nodes (node 0 is the root) followed by the
    retrieval slots; a slot whose template parent is -1 hangs off the root,
    any other slot off the node that holds its template parent."""
    nd = len(parent_draft)
    parent = list(int(p) for p in parent_draft)
    for p in tparent_stage:
        parent.append(0 if p < 0 else nd + int(p))
    return np.array(parent, np.int32)


CHECKPOINT_LAYERS = (0, 1, 5)


def cumulative_confidence(parent, conf):
    """depth int32 [N] (root 0) and cumulative confidence float32 [N]: the
    fp32 product of conf along the path, root excluded, root-to-node order
    (root: 1).  Parents precede their children (request-local indices)."""
    n = len(parent)
    depth = np.zeros(n, np.int32)
    c = np.ones(n, np.float32)
    for i in range(n):
        p = int(parent[i])
        if p >= 0:
            depth[i] = depth[p] + 1
            c[i] = np.float32(c[p] * np.float32(conf[i]))
    return depth, c


def stage_decision(parent, conf, node_off, tau):
    """Per request: best cumulative confidence at the checkpoint layers and the
    stage (first checkpoint whose best value is below its threshold; 3 if
    none).  Returns stage int32 [B], best float32 [B, 3]."""
    B = len(node_off) - 1
    stage = np.full(B, 3, np.int32)
    best = np.zeros((B, len(CHECKPOINT_LAYERS)), np.float32)
    for r in range(B):
        a, b = int(node_off[r]), int(node_off[r + 1])
        depth, c = cumulative_confidence(parent[a:b], conf[a:b])
        for j, L in enumerate(CHECKPOINT_LAYERS):
            at = c[depth == L + 1]
            best[r, j] = at.max() if at.size else np.float32(0.0)
        for j in range(len(CHECKPOINT_LAYERS)):
            if best[r, j] < np.float32(tau[j]):
                stage[r] = j
                break
    return stage, best


def graft_replace(parent, tok, conf, node_off, S, tau, attach, adj, tparent_bf, trank_bf):
    """Static-tree replacement (attach = 0: retrieval rooted at the current
    token) and Graft-TAIL (attach = 1: rooted at the deepest kept node, ties:
    larger cumulative confidence, then lower index).  Request r has S nodes
    (node 0 its root).  Returns tok_out, parent_out int32 [B, S] (-1 padded),
    n_kept int32 [B]; retrieval slot s follows the best-first template
    (tparent_bf, trank_bf), its first S - n_kept entries."""
    B = len(node_off) - 1
    tok_out = np.full((B, S), -1, np.int32)
    par_out = np.full((B, S), -1, np.int32)
    n_kept = np.zeros(B, np.int32)
    for r in range(B):
        a = int(node_off[r])
        p_loc = [int(x) for x in parent[a:a + S]]
        depth, c = cumulative_confidence(p_loc, conf[a:a + S])
        keep = [False] * S
        for i in range(S):
            keep[i] = i == 0 or (c[i] >= np.float32(tau) and keep[p_loc[i]])
        new = {}
        for i in range(S):
            if keep[i]:
                new[i] = len(new)
                tok_out[r, new[i]] = tok[a + i]
                par_out[r, new[i]] = -1 if i == 0 else new[p_loc[i]]
        nk = len(new)
        n_kept[r] = nk
        anchor = 0
        if attach == 1:
            for i in range(S):
                if keep[i] and (depth[i], c[i]) > (depth[anchor], c[anchor]):
                    anchor = i
        F = min(S - nk, len(tparent_bf))
        for s in range(F):
            tp = int(tparent_bf[s])
            src = int(tok[a + anchor]) if tp < 0 else int(tok_out[r, nk + tp])
            tok_out[r, nk + s] = adj[src, int(trank_bf[s])]
            par_out[r, nk + s] = new[anchor] if tp < 0 else nk + tp
    return tok_out, par_out, n_kept
