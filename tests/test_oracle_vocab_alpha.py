"""Pins for the oracle's vocab reductions and alpha = 1 - TV(p, q)."""
import numpy as np
import pytest
import scipy.special

import synth
from oracle import alpha as oal
from oracle import vocab as ovoc


def brute_topk(x, k):
    """Rank of i = number of entries that come before it in (value desc, index asc)."""
    V = len(x)
    rank = [sum(1 for j in range(V) if x[j] > x[i] or (x[j] == x[i] and j < i)) for i in range(V)]
    return [rank.index(t) for t in range(k)]


@pytest.mark.parametrize("seed", range(20))
def test_topk_and_argmax_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    V = int(rng.integers(8, 17))
    x = rng.integers(-3, 4, (3, V)).astype(np.float32)       # many ties
    k = int(rng.integers(1, min(V, 8) + 1))
    am, ti, tv, rm, _ = ovoc.argmax_topk(x, k)
    for r in range(3):
        assert ti[r].tolist() == brute_topk(x[r].tolist(), k)
        assert am[r] == min(i for i in range(V) if x[r, i] == x[r].max())
        assert ti[r, 0] == am[r]
        assert tv[r].tolist() == [x[r, i] for i in ti[r]]
        assert rm[r] == x[r].max()


def test_planted_argmax_recovered_fp32_and_bf16():
    d = synth.tiny_tree()
    am, ti, _, _, _ = ovoc.argmax_topk(d["logits"], 8)
    assert np.array_equal(am, d["planted"])
    b = synth.dcut_batch(B=3, V=5000, with_attention=False)
    am, ti, tv, _, _ = ovoc.argmax_topk(b["logits"], 8)
    assert np.array_equal(am, b["planted"])
    assert np.all(np.diff(tv, axis=1) <= 0)


def test_lse_matches_scipy_and_normalises():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((4, 3000)) * 3).astype(np.float32)
    _, _, _, _, lse = ovoc.argmax_topk(x, 0)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(x.astype(np.float64), axis=1), rtol=1e-13)
    for r in range(4):
        assert np.exp(x[r].astype(np.float64) - lse[r]).sum() == pytest.approx(1.0, abs=1e-12)


def test_alpha_identity_and_disjoint():
    rng = np.random.default_rng(2)
    lp = rng.standard_normal((3, 50))
    a, atv, _, _ = oal.tv_alpha(lp, lp)
    np.testing.assert_allclose(a, 1.0, atol=1e-13)
    # disjoint supports: -1e4 is an exact zero after exp in fp64
    lq = np.full((1, 6), -1e4)
    lp = np.full((1, 6), -1e4)
    lp[0, :3] = 0.0
    lq[0, 3:] = 0.0
    a, atv, _, _ = oal.tv_alpha(lp, lq)
    assert a[0] == 0.0 and atv[0] == pytest.approx(0.0, abs=1e-15)


def test_alpha_two_formulas_agree_and_bounded():
    d = synth.specopd_tree(prompt=8, response=40, n_anchor=4, W=5, V=3000, with_attention=False)
    a, atv, pre, pm = oal.tv_alpha(d["lp"], d["lq"], d["branch_off"], d["mass_tok"])
    np.testing.assert_allclose(a, atv, atol=1e-12)
    assert np.all((a >= 0) & (a <= 1))
    for b in range(4):
        run = pre[b * 5:(b + 1) * 5]
        assert np.all(np.diff(run) <= 0)
        assert run[0] == a[b * 5]
        assert run[-1] == pytest.approx(np.prod(a[b * 5:(b + 1) * 5]), rel=1e-14)


def test_alpha_two_point_closed_form():
    # p = (s, 1-s), q = (t, 1-t)  ->  alpha = 1 - |s - t|
    for s, t in [(0.3, 0.8), (0.5, 0.5), (0.99, 0.01), (0.2, 0.25)]:
        lp = np.log([[s, 1 - s]])
        lq = np.log([[t, 1 - t]])
        a, _, _, _ = oal.tv_alpha(lp, lq)
        assert a[0] == pytest.approx(1 - abs(s - t), abs=1e-14)


def test_softmax_mass_matches_scipy_and_sums_to_one():
    rng = np.random.default_rng(5)
    V = 40
    lp = rng.standard_normal((1, V)) * 2
    lq = rng.standard_normal((1, V))
    p = scipy.special.softmax(lp[0])
    total = 0.0
    for t in range(V):
        _, _, _, pm = oal.tv_alpha(lp, lq, mass_tok=np.array([t]))
        assert pm[0] == pytest.approx(p[t], rel=1e-13)
        total += pm[0]
    assert total == pytest.approx(1.0, abs=1e-13)
    one_hot = np.full((1, V), -1e4)
    one_hot[0, 7] = 0.0
    _, _, _, pm = oal.tv_alpha(one_hot, lq, mass_tok=np.array([7]))
    assert pm[0] == 1.0
