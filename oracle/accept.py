"""Greedy acceptance of the longest verified path.

Graft page section 2 (third gear): every candidate, draft or retrieved, is
held to the same verification rule, so the output equals plain decoding by
the target.  BlockPilot page introduction and SpecOPD page section 01: a
draft is accepted up to the first token that disagrees with the target, and
truncated there.  Graft page section 3: a larger tree never shortens the
longest accepted prefix.  SpecOPD page section 03 (worked example): with four
drafts, a wrong first token gives acceptance length 0; three right tokens
followed by a wrong one give 3.

Definition (greedy, temperature 0):
  acc(root)   = valid(root)
  acc(i)      = acc(parent(i)) and tok[i] == argmax[parent(i)] and valid(i)
  best        = the accepted node of largest depth, lowest index on ties
  accept_len  = depth(best)          (accepted draft tokens)
  path        = root .. best          (request-local indices, -1 padded)
  bonus       = argmax[best]          (the target's own next token)
  path_acc[i] = depth of the deepest accepted node on root..i (-1 if none):
                the acceptance length had the draft been the path to i.
A request whose root is not valid has best = bonus = -1, accept_len = -1.
"""
from __future__ import annotations

import numpy as np


def accept_longest_path(parent, tok, argmax, node_off, valid=None, max_depth=None):
    parent = np.asarray(parent)
    tok = np.asarray(tok)
    argmax = np.asarray(argmax)
    node_off = np.asarray(node_off)
    B = node_off.size - 1
    n = int(node_off[-1])
    accept_len = np.full(B, -1, np.int32)
    best_node = np.full(B, -1, np.int32)
    bonus = np.full(B, -1, np.int32)
    path_acc = np.full(n, -1, np.int32)
    paths = []
    for r in range(B):
        n0, n1 = int(node_off[r]), int(node_off[r + 1])
        N = n1 - n0
        children = [[] for _ in range(N)]
        roots = []
        for i in range(N):
            p = int(parent[n0 + i])
            (roots if p < 0 else children[p]).append(i)
        best, best_d = -1, -1
        # depth-first walk from every root over children in index order;
        # the stack carries (node, depth, accepted?, deepest accepted depth on the path)
        stack = [(i, 0, None, -1) for i in reversed(roots)]
        while stack:
            i, d, par_acc, deepest = stack.pop()
            ok_valid = valid is None or bool(valid[n0 + i])
            if par_acc is None:          # a root
                acc = ok_valid
            else:
                p = int(parent[n0 + i])
                acc = par_acc and ok_valid and int(tok[n0 + i]) == int(argmax[n0 + p])
            if acc:
                deepest = d
                if d > best_d or (d == best_d and i < best):
                    best, best_d = i, d
            path_acc[n0 + i] = deepest
            for c in reversed(children[i]):
                stack.append((c, d + 1, acc, deepest))
        path = []
        if best >= 0:
            j = best
            while j != -1:
                path.append(j)
                j = int(parent[n0 + j])
            path.reverse()
            best_node[r] = best
            accept_len[r] = best_d
            bonus[r] = int(argmax[n0 + best])
        paths.append(path)
    width = (max_depth + 1) if max_depth is not None else max([len(p) for p in paths] + [1])
    path_arr = np.full((B, width), -1, np.int32)
    for r, p in enumerate(paths):
        path_arr[r, :len(p)] = p[:width]
    return accept_len, best_node, path_arr, bonus, path_acc
