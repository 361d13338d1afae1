"""Pins for the oracle's next rows: Graft stage decision, static-tree
replacement and TAIL, D-cut expected tokens and budget choice."""
import json
import os

import numpy as np
import pytest

from oracle import dcut as odc
from oracle import graft as ogr


# ---------------------------------------------------------------- stage decision
def test_stage_decision_worked_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "graft_stage_decision.json")))
    par = np.array(g["parent"], np.int32)
    conf = np.array(g["conf"], np.float32)
    depth, c = ogr.cumulative_confidence(par, conf)
    assert depth.tolist() == g["depth"]
    assert c.tolist() == g["cumulative"]
    off = np.array([0, len(par)], np.int32)
    for case in g["cases"]:
        st, best = ogr.stage_decision(par, conf, off, case["tau"])
        assert best[0].tolist() == g["best_layers_0_1_5"]
        assert int(st[0]) == case["stage"], case


def test_stage_decision_chain_closed_form():
    # chain of 8 drafts at confidence 1/2: best at layer L is 2^-(L+1) exactly
    par = np.arange(-1, 8, dtype=np.int32)
    conf = np.full(9, 0.5, np.float32)
    st, best = ogr.stage_decision(par, conf, np.array([0, 9]), [0.5, 0.25, 2.0 ** -6])
    assert best[0].tolist() == [0.5, 0.25, 2.0 ** -6] and st[0] == 3
    st, _ = ogr.stage_decision(par, conf, np.array([0, 9]), [0.5, 0.25, 2.0 ** -5])
    assert st[0] == 2
    # a chain that stops at layer 3 never reaches checkpoint layer 5: best 0 there
    st, best = ogr.stage_decision(par[:5], conf[:5], np.array([0, 5]), [0.1, 0.1, 0.0])
    assert best[0, 2] == 0 and st[0] == 3
    st, _ = ogr.stage_decision(par[:5], conf[:5], np.array([0, 5]), [0.1, 0.1, 1e-9])
    assert st[0] == 2


def random_forest(rng, sizes):
    par, off = [], [0]
    for n in sizes:
        par += [-1] + [int(rng.integers(0, i)) for i in range(1, n)]
        off.append(off[-1] + n)
    return np.array(par, np.int32), np.array(off, np.int32)


def test_stage_decision_monotone_in_thresholds():
    rng = np.random.default_rng(11)
    par, off = random_forest(rng, rng.integers(1, 40, 30))
    conf = rng.uniform(0.05, 1.0, par.size).astype(np.float32)
    tau = rng.uniform(0, 0.6, 3)
    st, _ = ogr.stage_decision(par, conf, off, tau)
    st2, _ = ogr.stage_decision(par, conf, off, tau * 1.5)
    assert np.all(st2 <= st)   # stricter thresholds prune no later


# ------------------------------------------------------------ tree replacement
def chain_tree(tok, conf):
    n = len(tok)
    return np.arange(-1, n - 1, dtype=np.int32), np.asarray(tok, np.int32), np.asarray(conf, np.float32)


def test_replace_threshold_zero_keeps_the_tree():
    rng = np.random.default_rng(3)
    V, S = 500, 20
    par, off = random_forest(rng, [S, S])
    tok = rng.integers(0, V, par.size).astype(np.int32)
    conf = rng.uniform(0.1, 1, par.size).astype(np.float32)
    adj = rng.integers(0, V, (V, 8)).astype(np.int32)
    tp, tr = ogr.stage_template(60)
    t_out, p_out, nk = ogr.graft_replace(par, tok, conf, off, S, 0.0, 0, adj, tp, tr)
    assert nk.tolist() == [S, S]
    assert np.array_equal(t_out.reshape(-1), tok) and np.array_equal(p_out.reshape(-1), par)


def test_replace_everything_equals_plain_retrieval():
    # threshold above 1: only the root survives; the S - 1 retrieval slots are
    # exactly the (pinned) template retrieval with an (S - 1)-slot template
    rng = np.random.default_rng(4)
    V, S = 300, 25
    par, off = random_forest(rng, [S, S, S])
    tok = rng.integers(0, V, par.size).astype(np.int32)
    conf = np.ones(par.size, np.float32)
    adj = rng.integers(0, V, (V, 8)).astype(np.int32)
    tp, tr = ogr.stage_template(60)
    t_out, p_out, nk = ogr.graft_replace(par, tok, conf, off, S, 1.5, 0, adj, tp, tr)
    assert nk.tolist() == [1, 1, 1]
    tp24, tr24 = ogr.stage_template(S - 1)
    rtok, rpar, _ = ogr.retrieve(adj, tok[off[:-1]], np.zeros(3, np.int32), tp24, tr24,
                                 np.array([0, S - 1], np.int32), S - 1)
    assert np.array_equal(t_out[:, 1:], rtok)
    assert np.array_equal(p_out[:, 1:], np.where(rpar < 0, 0, rpar + 1))
    assert np.array_equal(t_out[:, 0], tok[off[:-1]])


def test_tail_keeps_the_confident_prefix():
    # 16-token block at dyadic confidences: cumulative 1/2, 1/4, 1/8, ... so a
    # threshold of 1/16 keeps exactly 4 drafts; the tail continues from the 4th
    V = 64
    adj = (np.arange(V)[:, None] * 7 + np.arange(8)[None, :]) % V
    par, tok, conf = chain_tree(np.arange(17) % V, [1.0] + [0.5] * 16)
    tp, tr = ogr.stage_template(60)
    t_out, p_out, nk = ogr.graft_replace(par, tok, conf, np.array([0, 17]), 17, 1 / 16, 1, adj, tp, tr)
    assert nk[0] == 5
    assert t_out[0, :5].tolist() == [0, 1, 2, 3, 4] and p_out[0, :5].tolist() == [-1, 0, 1, 2, 3]
    # first retrieval slot: rank-0 successor of the last kept token, under it
    assert p_out[0, 5] == 4 and t_out[0, 5] == adj[4, 0]
    # the greedy chain of the template: slot 1 is rank 0 under slot 0
    assert tp[1] == 0 and tr[1] == 0 and p_out[0, 6] == 5 and t_out[0, 6] == adj[adj[4, 0], 0]


def test_replace_structure_random():
    rng = np.random.default_rng(9)
    V, S = 1000, 60
    par, off = random_forest(rng, [S] * 6)
    tok = rng.integers(0, V, par.size).astype(np.int32)
    conf = rng.uniform(0.3, 1, par.size).astype(np.float32)
    adj = rng.integers(0, V, (V, 8)).astype(np.int32)
    tp, tr = ogr.stage_template(60)
    for attach in (0, 1):
        t_out, p_out, nk = ogr.graft_replace(par, tok, conf, off, S, 0.5, attach, adj, tp, tr)
        for r in range(6):
            assert p_out[r, 0] == -1 and np.all(t_out[r] >= 0)          # S slots filled
            assert np.all(p_out[r, 1:] < np.arange(1, S))               # parents precede
            assert np.all(p_out[r, 1:] >= 0)
            d, c = ogr.cumulative_confidence(par[off[r]:off[r + 1]], conf[off[r]:off[r + 1]])
            keep = (c >= np.float32(0.5))
            # kept = nodes whose whole path clears the threshold
            ok = [True] * S
            for i in range(1, S):
                ok[i] = bool(keep[i]) and ok[par[off[r] + i]]
            assert nk[r] == sum(ok)


# ------------------------------------------------- D-cut expected tokens, rho*
def test_expected_tokens_closed_forms():
    B, D = 5, 15
    conf = np.full((B, D), 0.5, np.float32)
    s, keep, *_ = odc.select(conf, [0.25, 0.5, 1.0])
    E = odc.expected_tokens(s, keep)
    assert E[-1] == B * (2 - 2.0 ** -D)            # sum_j 2^-j, j = 0..D, per request
    assert np.all(np.diff(E) >= 0)
    s1, keep1, *_ = odc.select(np.ones((B, D), np.float32), [0.25, 0.5, 0.75, 1.0])
    assert odc.expected_tokens(s1, keep1).tolist() == [odc.budget(r, B * (D + 1)) for r in (0.25, 0.5, 0.75, 1.0)]


def test_choose_rho_worked_example():
    # gains 30, 50, 62, 70 tokens against step costs 1.0, 1.4, 1.9, 2.6 (ms):
    # ratios 30, 35.7, 32.6, 26.9 -> the second budget
    assert odc.choose_rho([30.0, 50.0, 62.0, 70.0], [1.0, 1.4, 1.9, 2.6]) == 1
    assert odc.choose_rho([10.0, 20.0], [1.0, 2.0]) == 0     # tie: lowest index
