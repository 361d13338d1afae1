"""Pins for the oracle's acceptance and Graft table routines."""
import itertools
import json
import os

import numpy as np
import pytest

import synth
from oracle import accept as oacc
from oracle import graft as ogr


def test_worked_example_golden(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "specopd_worked_example.json")))
    for case in g["cases"]:
        correct = case["draft_correct"]
        n = len(correct) + 1
        parent = np.arange(-1, n - 1, dtype=np.int32)
        argmax = np.arange(100, 100 + n, dtype=np.int32)      # target's choice at each node
        tok = np.zeros(n, np.int32)
        for j, ok in enumerate(correct, start=1):
            tok[j] = argmax[j - 1] if ok else 7
        al, best, path, bonus, _ = oacc.accept_longest_path(parent, tok, argmax, [0, n])
        assert al[0] == case["accept_len"], case["name"]
        assert bonus[0] == argmax[case["accept_len"]]
        assert path[0, :al[0] + 1].tolist() == list(range(al[0] + 1))


def brute_accept(parent, tok, argmax, valid):
    """Enumerate every node's root path; accepted iff every step matches."""
    n = len(parent)
    acc, depth = [], []
    for i in range(n):
        path = [i]
        while parent[path[-1]] >= 0:
            path.append(parent[path[-1]])
        path.reverse()
        ok = all(valid[j] for j in path) and all(
            tok[path[t]] == argmax[path[t - 1]] for t in range(1, len(path)))
        acc.append(ok)
        depth.append(len(path) - 1)
    cands = [(depth[i], -i) for i in range(n) if acc[i]]
    if not cands:
        return -1, -1, acc, depth
    d, negi = max(cands)
    return d, -negi, acc, depth


@pytest.mark.parametrize("seed", range(40))
def test_accept_brute_force(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 9))
    parent = np.full(n, -1, np.int32)
    for i in range(1, n):
        parent[i] = -1 if rng.random() < 0.15 else rng.integers(0, i)
    V = 3
    tok = rng.integers(0, V, n).astype(np.int32)
    argmax = rng.integers(0, V, n).astype(np.int32)
    valid = (rng.random(n) < 0.85).astype(np.uint8)
    al, best, path, bonus, pacc = oacc.accept_longest_path(parent, tok, argmax, [0, n], valid)
    d, b, acc, depth = brute_accept(parent, tok, argmax, valid)
    assert al[0] == d and best[0] == b
    if b >= 0:
        assert bonus[0] == argmax[b]
        p = path[0][path[0] >= 0].tolist()
        assert p[-1] == b and len(p) == d + 1 and (parent[p[0]] == -1)
    for i in range(n):
        # path_acc: deepest accepted node on i's root path
        chain = [i]
        while parent[chain[-1]] >= 0:
            chain.append(parent[chain[-1]])
        best_d = max([depth[j] for j in chain if acc[j]], default=-1)
        assert pacc[i] == best_d


def test_chain_counts_leading_matches():
    rng = np.random.default_rng(9)
    for _ in range(50):
        n = 16
        parent = np.arange(-1, n - 1, dtype=np.int32)
        argmax = rng.integers(0, 4, n).astype(np.int32)
        tok = rng.integers(0, 4, n).astype(np.int32)
        match = [tok[j] == argmax[j - 1] for j in range(1, n)]
        lead = next((j for j, m in enumerate(match) if not m), n - 1)
        al, *_ = oacc.accept_longest_path(parent, tok, argmax, [0, n])
        assert al[0] == lead


@pytest.mark.parametrize("seed", range(10))
def test_superset_never_shortens(seed):
    """Graft page section 3: a tree containing another accepts at least as much."""
    d = synth.tiny_tree(step=seed, N=60)
    parent, tok = d["parent"], d["tok"]
    argmax = d["planted"]
    prev = -1
    for n in range(1, 61, 3):
        al, *_ = oacc.accept_longest_path(parent[:n], tok[:n], argmax[:n], [0, n])
        assert al[0] >= prev
        prev = al[0]


def test_acceptance_ignores_provenance_and_multirequest_offsets():
    d = synth.tiny_tree(N=20)
    one = oacc.accept_longest_path(d["parent"], d["tok"], d["planted"], [0, 20])
    two = oacc.accept_longest_path(np.tile(d["parent"], 2), np.tile(d["tok"], 2),
                                   np.tile(d["planted"], 2), [0, 20, 40])
    assert two[0].tolist() == [one[0][0]] * 2 and two[1].tolist() == [one[1][0]] * 2


# ----------------------------------------------------------------- Graft table
def test_adj_update_semantics():
    rng = np.random.default_rng(0)
    V, k = 50, 4
    adj = rng.integers(0, V, (V, k)).astype(np.int32)
    before = adj.copy()
    tok = np.array([3, 9, 3, 11, 9], np.int32)
    topk = rng.integers(0, V, (5, 6)).astype(np.int32)
    valid = np.array([1, 1, 1, 1, 0], np.uint8)
    ogr.adj_update(adj, tok, topk, valid)
    assert adj[3].tolist() == topk[2, :k].tolist()          # last writer wins
    assert adj[9].tolist() == topk[1, :k].tolist()          # invalid node 4 skipped
    assert adj[11].tolist() == topk[3, :k].tolist()
    untouched = [t for t in range(V) if t not in (3, 9, 11)]
    assert np.array_equal(adj[untouched], before[untouched])
    again = adj.copy()
    ogr.adj_update(again, tok, topk, valid)
    assert np.array_equal(again, adj)                       # idempotent


def test_stage_templates_match_budget_golden(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "graft_stage_budget.json")))
    tp, tr, off = ogr.stage_templates(k=g["best_width"], max_depth=g["best_depth"])
    assert np.diff(off).tolist() == g["retrieval"]
    assert [g["budget"] - s for s in g["retrieval"]] == g["draft"]
    for st in range(4):
        p = tp[off[st]:off[st + 1]]
        r = tr[off[st]:off[st + 1]]
        S = len(p)
        if S == 0:
            continue
        assert np.all(p < np.arange(S))                      # parents first
        assert np.all((r >= 0) & (r < g["best_width"]))
        depth = np.zeros(S, int)
        top = np.zeros(S, int)
        for s in range(S):
            depth[s] = 1 if p[s] < 0 else depth[p[s]] + 1
            top[s] = r[s] if p[s] < 0 else top[p[s]]
        assert depth.max() <= g["best_depth"]
        # asymmetric: the rank-0 successor's subtree is the largest and deepest
        sizes = [int((top == t).sum()) for t in range(g["best_width"])]
        assert sizes[0] == max(sizes) and sizes[0] > S // 2
        assert depth[top == 0].max() == depth.max()
        # smaller stages are prefixes of larger ones (same best-first order)
        if st > 0:
            assert np.array_equal(p, tp[:S]) and np.array_equal(r, tr[:S])
        # no two slots repeat the same (parent, rank) edge
        assert len(set(zip(p.tolist(), r.tolist()))) == S


def test_retrieve_identity_successor_closed_form():
    V, k = 97, 8
    adj = np.array([[(t + r + 1) % V for r in range(k)] for t in range(V)], np.int32)
    tp, tr, off = ogr.stage_templates()
    roots = np.array([0, 5, 96, 50], np.int32)
    stage = np.array([0, 1, 2, 3], np.int32)
    rtok, rpar, ns = ogr.retrieve(adj, roots, stage, tp, tr, off, 52)
    assert ns.tolist() == [52, 36, 20, 0]
    for b in range(4):
        s0 = off[stage[b]]
        for s in range(ns[b]):
            total, j = 0, s
            while j >= 0:
                total += tr[s0 + j] + 1
                j = tp[s0 + j]
            assert rtok[b, s] == (roots[b] + total) % V
            assert rpar[b, s] == tp[s0 + s]
        assert np.all(rtok[b, ns[b]:] == -1)


def test_retrieve_brute_force_tiny():
    rng = np.random.default_rng(4)
    V, k = 6, 3
    adj = rng.integers(0, V, (V, k)).astype(np.int32)
    tp, tr, off = ogr.stage_templates(k=k, max_depth=3, slots=(10, 4))
    rtok, _, _ = ogr.retrieve(adj, np.array([2, 4]), np.array([0, 1]), tp, tr, off, 10)
    for b, (root, st) in enumerate([(2, 0), (4, 1)]):
        for s in range(off[st + 1] - off[st]):
            ranks, j = [], s
            while j >= 0:
                ranks.append(tr[off[st] + j])
                j = tp[off[st] + j]
            t = root
            for r in reversed(ranks):
                t = adj[t, r]
            assert rtok[b, s] == t


def test_template_enumeration_brute_force_small():
    """Best-first order equals a full sort of all rank paths by exact weight."""
    from fractions import Fraction
    k, depth, S = 3, 3, 20
    paths = [p for L in range(1, depth + 1) for p in itertools.product(range(k), repeat=L)]
    w = lambda p: np.prod([Fraction(9, 10) * Fraction(2, 5) ** r for r in p])
    paths.sort(key=lambda p: (-w(p), p))
    tp, tr = ogr.stage_template(S, k=k, max_depth=depth)
    slot = {p: i for i, p in enumerate(paths[:S])}
    for i, p in enumerate(paths[:S]):
        assert tr[i] == p[-1]
        assert tp[i] == (slot[p[:-1]] if len(p) > 1 else -1)
