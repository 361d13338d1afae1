"""Pins for the oracle's D-cut selection and BlockPilot predictor."""
import json
import os

import numpy as np
import pytest

import synth
from oracle import accept as oacc
from oracle import dcut as odc
from oracle import mlp as omlp


def test_budget_golden(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "dcut_budget.json")))
    total = g["B"] * (g["D"] + 1)
    assert [odc.budget(r, total) for r in g["rho"]] == g["K"]


def test_selection_invariants_on_workload():
    d = synth.dcut_batch(with_attention=False, with_logits=False)
    s, keep, keep_len, pack_off, pack_idx = odc.select(d["conf"], d["rho"])
    B, N = s.shape
    assert np.all(s[:, 0] == 1.0) and np.all(np.diff(s, axis=1) <= 0)
    for a, rho in enumerate(d["rho"]):
        K = odc.budget(rho, B * N)
        assert keep[a].sum() == K
        for r in range(B):
            L = keep_len[a, r]
            assert keep[a, r, :L].all() and not keep[a, r, L:].any()   # prefix-closed
        assert pack_off[a, -1] == K
        assert pack_idx[a, :K].tolist() == np.nonzero(keep[a].reshape(-1))[0].tolist()
        if a:
            assert np.all(keep[a - 1] <= keep[a])                         # monotone in rho
    assert keep[-1].all()                                                 # rho = 1 keeps all


def brute_select(s, K):
    B, N = s.shape
    items = [(r, j) for r in range(B) for j in range(N)]
    rank = {}
    for (r, j) in items:
        rank[(r, j)] = sum(1 for (r2, j2) in items
                           if s[r2, j2] > s[r, j] or (s[r2, j2] == s[r, j] and (r2, j2) < (r, j)))
    return np.array([[1 if rank[(r, j)] < K else 0 for j in range(N)] for r in range(B)], np.uint8)


@pytest.mark.parametrize("seed", range(8))
def test_selection_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    B, D = int(rng.integers(1, 5)), int(rng.integers(1, 6))
    conf = rng.choice(np.array([1.0, 0.5, 0.25], np.float32), (B, D))   # exact ties
    rhos = [0.1, 0.3, 0.5, 0.9]
    s, keep, *_ = odc.select(conf, rhos)
    for a, rho in enumerate(rhos):
        assert np.array_equal(keep[a], brute_select(s, odc.budget(rho, s.size)))


def test_prefix_scores_are_sequential_fp32():
    conf = np.array([[0.1, 0.2, 0.3, 0.7]], np.float32)
    s = odc.prefix_scores(conf)
    run = np.float32(1.0)
    for j in range(4):
        run = np.float32(run * conf[0, j])
        assert s[0, j + 1] == run


def test_prefix_survival_monte_carlo():
    """BlockPilot page section 8 / D-cut page section 2: with independent
    per-position survival c_j, E[accepted] = sum_k prod_{j<=k} c_j."""
    B, D = 400, 15
    d = synth.dcut_batch(B=B, D=D, V=10**6, with_attention=False, with_logits=False)
    s = odc.prefix_scores(d["conf"]).astype(np.float64)
    N = D + 1
    # the workload plants argmax; the draft matches it with probability conf
    al, *_ = oacc.accept_longest_path(d["parent"], d["tok"], d["planted"], d["node_off"])
    expect = s[:, 1:].sum(axis=1)
    diff = al - expect
    z = diff.mean() / (diff.std(ddof=1) / np.sqrt(B))
    assert abs(z) < 4.0, (al.mean(), expect.mean())


# ---------------------------------------------------------------- BlockPilot
def test_zero_weights_pick_lowest_index(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "blockpilot_window.json")))
    rng = np.random.default_rng(0)
    logits = rng.standard_normal((3, 100))
    z, choice, block = omlp.blockpilot(logits, np.zeros((100, 8)), np.zeros(8), np.zeros((8, 7)),
                                       np.zeros(7), block=g["B"])
    assert np.all(z == 0) and np.all(choice == 0) and np.all(block == g["sizes"][0])
    assert g["B"] - 3 == g["sizes"][0] and g["B"] + 3 == g["sizes"][-1]


def test_mlp_closed_form_probability_readout():
    """W1 = identity on the first H tokens, W2 = identity: z = probabilities."""
    rng = np.random.default_rng(1)
    V, H = 30, 7
    logits = rng.standard_normal((4, V)) * 2
    W1 = np.zeros((V, H))
    W1[:H, :H] = np.eye(H)
    z, choice, block = omlp.blockpilot(logits, W1, np.zeros(H), np.eye(H), np.zeros(H))
    p = np.exp(logits - logits.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    np.testing.assert_allclose(z, p[:, :H], rtol=1e-13)
    assert choice.tolist() == np.argmax(p[:, :H], axis=1).tolist()
    assert block.tolist() == (13 + choice).tolist()


def test_mlp_relu_and_bias():
    V = 5
    logits = np.zeros((1, V))                      # uniform: x = 0.2 each
    W1 = np.array([[1.0, -1.0]] * V)               # h_pre = (1, -1) + b1
    b1 = np.array([0.5, 0.25])
    W2 = np.array([[1.0, 0.0, 2.0], [10.0, 10.0, 10.0]])
    z, choice, _ = omlp.blockpilot(logits, W1, b1, W2, np.array([0.0, 3.0, 0.0]), block=2)
    # h = relu(1.5, -0.75) = (1.5, 0)
    np.testing.assert_allclose(z[0], [1.5, 3.0, 3.0], rtol=1e-15)
    assert choice[0] == 1                          # tie 3.0 / 3.0 -> lowest index


def test_budget_rounds_half_up():
    """Reading of the D-cut budget: K = rho * B * (D+1) rounded to the nearest
    integer, halves up (the page's ratios give whole numbers at 64 x 16)."""
    assert odc.budget(0.25, 6) == 2      # 1.5  -> 2
    assert odc.budget(0.1, 16) == 2      # 1.6  -> 2
    assert odc.budget(0.5, 7) == 4       # 3.5  -> 4
    assert odc.budget(0.75, 5) == 4      # 3.75 -> 4
    assert odc.budget(0.25, 5) == 1      # 1.25 -> 1
