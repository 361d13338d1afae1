"""Pins for the oracle's T = 1 rejection-sampling verification."""
import numpy as np
import pytest

from oracle import sampling as osm


def first_token_frequencies(pl, ql, parent, n_sib, trials, seed):
    """Draft the children of each node i.i.d. from that node's draft
    distribution (as the scheme assumes), verify, and count the first emitted
    token: the accepted first draft, else the bonus token."""
    rng = np.random.default_rng(seed)
    V = pl.shape[1]
    q = np.exp(ql - ql.max(axis=1, keepdims=True))
    q /= q.sum(axis=1, keepdims=True)
    cnt = np.zeros(V)
    n = len(parent)
    for _ in range(trials):
        tok = np.zeros(n, np.int64)
        for i in range(1, n):
            tok[i] = rng.choice(V, p=q[parent[i]])
        acc, _, path, bonus, _, _ = osm.rejection_verify(parent, tok, pl, ql, np.array([0, n]), rng.random(n),
                                                      rng.random(1), n)
        cnt[tok[path[0, 1]] if acc[0] >= 1 else bonus[0]] += 1
    return cnt / trials


@pytest.mark.parametrize("shape", ["chain", "siblings"])
def test_first_token_follows_the_target(shape):
    # the defining property of lossless verification: whatever the draft, the
    # first emitted token is distributed as the target's softmax at the root
    p0 = np.array([0.1, 0.2, 0.3, 0.4])
    pl = np.log(np.array([p0, [0.25] * 4, [0.7, 0.1, 0.1, 0.1], [0.1, 0.6, 0.2, 0.1]]))
    ql = np.log(np.array([[0.4, 0.3, 0.2, 0.1], [0.1, 0.1, 0.1, 0.7], [0.25] * 4, [0.5, 0.2, 0.2, 0.1]]))
    parent = np.array([-1, 0, 1]) if shape == "chain" else np.array([-1, 0, 0, 0])
    f = first_token_frequencies(pl[:len(parent)], ql[:len(parent)], parent, 0, 20000, 5)
    sigma = np.sqrt(p0 * (1 - p0) / 20000)
    assert np.all(np.abs(f - p0) < 4.5 * sigma), (f, p0)


def test_identical_distributions_accept_every_first_child():
    rng = np.random.default_rng(1)
    n, V = 12, 50
    parent = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, n)])
    lg = rng.standard_normal((n, V))
    tok = rng.integers(0, V, n)
    acc, best, path, _, _, _ = osm.rejection_verify(parent, tok, lg, lg, np.array([0, n]), rng.random(n) * 0.999,
                                                 np.array([0.5]), n)
    # expected: follow the lowest-index child at every step down to a leaf
    cur, d = 0, 0
    while True:
        kids = [i for i in range(n) if parent[i] == cur]
        if not kids:
            break
        cur, d = kids[0], d + 1
    assert acc[0] == d and best[0] == cur


def test_one_hot_draft_accepts_with_the_target_probability():
    V = 5
    p = np.array([0.05, 0.15, 0.3, 0.2, 0.3])
    pl = np.log(np.array([p, p]))
    ql = np.array([[-60.0, -60.0, 0.0, -60.0, -60.0], [0.0] * V])   # the draft is sure of token 2
    parent, tok = np.array([-1, 0]), np.array([0, 2])
    for u, want in ((0.29, 1), (0.31, 0)):
        acc, _, _, _, _, _ = osm.rejection_verify(parent, tok, pl, ql, np.array([0, 2]), np.array([0.0, u]),
                                               np.array([0.5]), 1)
        assert acc[0] == want
    # after that rejection the residual is p without token 2, renormalised:
    # cdf 0.05/0.7, 0.2/0.7, (same), 0.4/0.7, 1 = 0.071, 0.286, 0.286, 0.571, 1
    for uf, want in ((0.25, 1), (0.3, 3), (0.6, 4), (0.05, 0)):
        _, _, _, bonus, _, _ = osm.rejection_verify(parent, tok, pl, ql, np.array([0, 2]), np.array([0.0, 0.9]),
                                                 np.array([uf]), 1)
        assert bonus[0] == want


def zero_residual_case(V=64):
    """A root whose target and draft distributions differ only below the
    rounding of the normaliser: target logits (0, -40), draft (0, -39), the
    other tokens at -1000 (exp underflows to exactly 0).  Then p(0) = q(0) = 1
    exactly, p(1) = e^-40 < q(1) = e^-39, so drafting token 1 is rejected
    with probability 1 - e^-1 and the residual max(0, p - q) is exactly 0
    (in float64 and in float32 alike).  The scheme is then undefined (0/0);
    the reading used: continue with the target softmax.  Children of the
    root: node 1 drafts token 1, node 2 (only in the two-child tree) drafts
    token 0; node 2's target puts all its mass on token 2."""
    pl = np.full((3, V), -1000.0)
    ql = np.full((3, V), -1000.0)
    pl[0, :2] = (0.0, -40.0)
    ql[0, :2] = (0.0, -39.0)
    pl[1:, 2] = 0.0
    ql[1:, 2] = 0.0
    return pl, ql


def test_zero_residual_continues_with_the_target_softmax():
    pl, ql = zero_residual_case()
    # one child, rejected (u = 0.5 > e^-1): the bonus token comes from the
    # target softmax at the root, (1, e^-40, 0, ...): token 0 for any u < 1
    for uf in (0.001, 0.5, 0.999):
        acc, best, _, bonus, trace, finals = osm.rejection_verify(
            np.array([-1, 0]), np.array([0, 1]), pl[:2], ql[:2], np.array([0, 2]), np.array([0.0, 0.5]),
            np.array([uf]), 1)
        assert acc[0] == 0 and best[0] == 0 and bonus[0] == 0
        assert abs(trace[0][2] - np.exp(-1.0)) < 1e-12
        assert np.all(np.isfinite(finals[0])) and finals[0][0] == 1.0
    # two children: after the zero-residual rejection of node 1, node 2
    # (token 0) meets p'(0) = q(0) = 1 and is accepted whatever its uniform;
    # the bonus then comes from node 2's target: token 2
    acc, best, path, bonus, trace, _ = osm.rejection_verify(
        np.array([-1, 0, 0]), np.array([0, 1, 0]), pl, ql, np.array([0, 3]), np.array([0.0, 0.5, 0.999]),
        np.array([0.3]), 2)
    assert acc[0] == 1 and best[0] == 2 and bonus[0] == 2
    assert list(path[0]) == [0, 2, -1]
    assert trace[1][2] == 1.0
