"""Parity of the next rows' kernels with the oracle: Graft stage decision,
static-tree replacement and TAIL, D-cut expected tokens and budget choice."""
import json
import os

import numpy as np
import pytest

import synth
from gpu_util import dev, host, sync
from oracle import dcut as odc
from oracle import graft as ogr

pytestmark = pytest.mark.gpu


def forest(rng, sizes, depth_bias=0.0):
    par, off = [], [0]
    for n in sizes:
        loc = [-1]
        for i in range(1, n):
            lo = max(0, int(i * depth_bias))
            loc.append(int(rng.integers(lo, i)))
        par += loc
        off.append(off[-1] + n)
    return np.array(par, np.int32), np.array(off, np.int32)


# ---------------------------------------------------------------- stage decision
def check_stage(tv, par, conf, off, tau):
    st, best, err = tv.graft_stage_decide(dev(par), dev(conf), dev(off), tau, max_nodes=int(np.diff(off).max()))
    sync()
    rst, rbest = ogr.stage_decision(par, conf, off, tau)
    assert np.array_equal(host(best), rbest)          # same fp32 products, same order
    assert np.array_equal(host(st), rst)
    assert host(err)[0] == 0
    return host(st)


def test_stage_decide_worked_example(tv, golden_dir):
    g = json.load(open(os.path.join(golden_dir, "graft_stage_decision.json")))
    par, conf = np.array(g["parent"], np.int32), np.array(g["conf"], np.float32)
    for case in g["cases"]:
        st = check_stage(tv, par, conf, np.array([0, len(par)], np.int32), case["tau"])
        assert st[0] == case["stage"]


@pytest.mark.parametrize("seed", range(4))
def test_stage_decide_random_forests(tv, seed):
    rng = np.random.default_rng(seed)
    sizes = rng.integers(1, 120, 40)
    sizes[0] = 1                                       # a request with only its root
    par, off = forest(rng, sizes, depth_bias=0.6)      # deep trees reach layer 5
    conf = rng.uniform(0.2, 1.0, par.size).astype(np.float32)
    st = check_stage(tv, par, conf, off, rng.uniform(0.0, 0.6, 3).tolist())
    assert set(st.tolist()) <= {0, 1, 2, 3}


def test_stage_decide_deep_chain(tv):
    n = 1024
    par = np.arange(-1, n - 1, dtype=np.int32)
    conf = np.full(n, 0.999, np.float32)
    check_stage(tv, par, conf, np.array([0, n], np.int32), [0.5, 0.5, 0.99])


# ------------------------------------------------------------ tree replacement
def check_replace(tv, par, tok, conf, S, tau, attach, adj, tp, tr):
    B = tok.size // S
    off = np.arange(B + 1, dtype=np.int32) * S
    to, po, nk, err = tv.graft_replace(dev(par), dev(tok), dev(conf), S, tau, attach, dev(adj), dev(tp), dev(tr))
    sync()
    rto, rpo, rnk = ogr.graft_replace(par, tok, conf, off, S, tau, attach, adj, tp, tr)
    assert np.array_equal(host(nk), rnk)
    assert np.array_equal(host(to), rto)
    assert np.array_equal(host(po), rpo)
    assert host(err)[0] == 0
    return rnk


@pytest.mark.parametrize("tau", [0.0, 0.3, 0.6, 1.5])
def test_replace_static_trees(tv, tau):
    rng = np.random.default_rng(int(tau * 10))
    B, S, V = 16, 60, synth.QWEN3_VOCAB
    par, _ = forest(rng, [S] * B, depth_bias=0.3)
    tok = rng.integers(0, V, B * S).astype(np.int32)
    conf = rng.uniform(0.3, 1.0, B * S).astype(np.float32)
    adj = synth.successor_table(2, V, 8)
    tp, tr = ogr.stage_template(60)
    nk = check_replace(tv, par, tok, conf, S, tau, 0, adj, tp, tr)
    if tau == 0.0:
        assert np.all(nk == S)
    if tau > 1:
        assert np.all(nk == 1)


@pytest.mark.parametrize("tau", [0.05, 0.2, 0.5])
def test_replace_tail_of_block_drafts(tv, tau):
    # DFlash-style 16-token blocks: chains of root + 16 drafts
    rng = np.random.default_rng(7)
    B, S, V = 32, 17, 5000
    par = np.tile(np.arange(-1, S - 1, dtype=np.int32), B)
    tok = rng.integers(0, V, B * S).astype(np.int32)
    conf = rng.beta(4, 1.5, B * S).astype(np.float32)
    adj = rng.integers(0, V, (V, 8)).astype(np.int32)
    tp, tr = ogr.stage_template(60)
    check_replace(tv, par, tok, conf, S, tau, 1, adj, tp, tr)


def test_replace_short_template_pads(tv):
    rng = np.random.default_rng(8)
    B, S, V = 4, 40, 300
    par, _ = forest(rng, [S] * B)
    tok = rng.integers(0, V, B * S).astype(np.int32)
    conf = np.full(B * S, 0.5, np.float32)
    adj = rng.integers(0, V, (V, 8)).astype(np.int32)
    tp, tr = ogr.stage_template(10)                    # fewer slots than freed
    check_replace(tv, par, tok, conf, S, 0.9, 0, adj, tp, tr)


# ------------------------------------------------- D-cut expected tokens, rho*
@pytest.mark.parametrize("which", ["workload", "ones"])
def test_choose_rho(tv, which):
    if which == "workload":
        conf = synth.dcut_batch(with_attention=False, with_logits=False)["conf"]
        cost = [1.0, 1.35, 1.8, 2.4]
    else:
        conf = np.ones((20, 7), np.float32)
        cost = [1.0, 1.9, 2.95, 3.9]
    rhos = list(synth.DCUT_RHOS)
    s, keep, *_ = tv.dcut_select(dev(conf), rhos)
    E, rs = tv.dcut_choose_rho(s, keep, cost)
    sync()
    rs_, rkeep, *_ = odc.select(conf, rhos)
    rE = odc.expected_tokens(rs_, rkeep)
    np.testing.assert_allclose(host(E), rE, rtol=1e-11)          # 2^-50 fixed point, <= 8192 terms
    ratios = np.sort(rE / np.array(cost))
    assert ratios[-1] - ratios[-2] > 1e-9 * ratios[-1]          # a unique best budget
    assert host(rs)[0] == odc.choose_rho(rE, cost)


# ------------------------------------------------ T = 1 rejection sampling
def sampling_case(seed, sizes, V, dtype="bf16"):
    """Trees whose children are drawn from the draft softmax of their parent
    (as the scheme assumes); target logits correlated with the draft's so
    that paths of several accepts occur."""
    from oracle import sampling as osm
    rng = np.random.default_rng(seed)
    par, off = forest(rng, sizes, depth_bias=0.5)
    n = par.size
    base = rng.standard_normal((n, V)).astype(np.float32) * 2.0
    ql = base + rng.standard_normal((n, V)).astype(np.float32) * 0.5
    pl = base + rng.standard_normal((n, V)).astype(np.float32) * 0.5
    if dtype == "bf16":
        pl, ql = synth.bf16_bits(pl), synth.bf16_bits(ql)
        pf, qf = osm._row(pl, slice(None)), osm._row(ql, slice(None))
    else:
        pf, qf = pl, ql
    tok = np.zeros(n, np.int32)
    for r in range(len(sizes)):
        a = off[r]
        for i in range(1, sizes[r]):
            q = osm._softmax64(qf[a + par[a + i]])
            tok[a + i] = rng.choice(V, p=q)
    u = rng.random(n).astype(np.float32)
    uf = rng.random(len(sizes)).astype(np.float32)
    # keep every uniform that decides a test at least 1e-3 from its threshold
    for _ in range(20):
        res = osm.rejection_verify(par, tok, pl, ql, off, u, uf, int(np.diff(off).max()) - 1)
        close = [(r, c) for r, c, ratio in res[4] if abs(float(u[off[r] + c]) - ratio) < 1e-3]
        if not close:
            break
        for r, c in close:
            u[off[r] + c] = np.float32(rng.random())
    return par, off, tok, pl, ql, u, uf, res


@pytest.mark.parametrize("seed,dtype", [(0, "bf16"), (1, "bf16"), (2, "f32")])
def test_rejection_sampling_matches_oracle(tv, seed, dtype):
    V = 3000 if dtype == "f32" else 5003
    sizes = [1, 2, 9, 40, 17, 60, 25, 3]
    par, off, tok, pl, ql, u, uf, (racc, rbest, rpath, rbonus, _, finals) = sampling_case(seed, sizes, V, dtype)
    max_depth = int(np.diff(off).max()) - 1
    acc, best, path, bonus = tv.accept_rejection_sampling(dev(par), dev(tok), dev(pl), dev(ql), dev(off), dev(u),
                                                          dev(uf), max_depth=max_depth)
    sync()
    assert np.array_equal(host(acc), racc)
    assert np.array_equal(host(best), rbest)
    assert np.array_equal(host(path), rpath)
    # the bonus token: equal, or u_final within 1e-5 of the CDF step between
    # the two choices (fp32 exponentials against the float64 oracle)
    for r, j in enumerate(host(bonus)):
        if j != rbonus[r]:
            cdf = np.cumsum(finals[r])
            lo = cdf[j - 1] if j > 0 else 0.0
            assert lo - 1e-5 <= uf[r] * cdf[-1] <= cdf[j] + 1e-5, (r, j, rbonus[r])
    assert np.mean(host(acc)) > 0.3                    # paths with accepts occur


def test_rejection_sampling_full_vocabulary(tv):
    # the launch configuration the benchmark times: V = 151936 bf16 rows, one
    # 8-CTA cluster per request, 16-node trees
    V = synth.QWEN3_VOCAB
    sizes = [16, 16, 16, 16]
    par, off, tok, pl, ql, u, uf, (racc, rbest, rpath, rbonus, _, finals) = sampling_case(7, sizes, V, "bf16")
    acc, best, path, bonus = tv.accept_rejection_sampling(dev(par), dev(tok), dev(pl), dev(ql), dev(off), dev(u),
                                                          dev(uf), max_depth=15)
    sync()
    assert np.array_equal(host(acc), racc)
    assert np.array_equal(host(best), rbest)
    assert np.array_equal(host(path), rpath)
    for r, j in enumerate(host(bonus)):
        if j != rbonus[r]:
            cdf = np.cumsum(finals[r])
            lo = cdf[j - 1] if j > 0 else 0.0
            assert lo - 1e-5 <= uf[r] * cdf[-1] <= cdf[j] + 1e-5, (r, j, rbonus[r])


def test_rejection_sampling_identical_distributions(tv):
    # draft = target: every first child is accepted, down to a leaf
    rng = np.random.default_rng(5)
    V = 2000
    par, off = forest(rng, [30, 30, 30], depth_bias=0.4)
    lg = synth.bf16_bits(rng.standard_normal((par.size, V)).astype(np.float32))
    tok = rng.integers(0, V, par.size).astype(np.int32)
    u = (rng.random(par.size) * 0.999).astype(np.float32)
    uf = rng.random(3).astype(np.float32)
    acc, best, path, bonus = tv.accept_rejection_sampling(dev(par), dev(tok), dev(lg), dev(lg), dev(off), dev(u),
                                                          dev(uf), max_depth=29)
    sync()
    for r in range(3):
        loc = par[off[r]:off[r + 1]]
        cur, d = 0, 0
        while True:
            kids = [i for i in range(len(loc)) if loc[i] == cur]
            if not kids:
                break
            cur, d = kids[0], d + 1
        assert host(acc)[r] == d and host(best)[r] == cur


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rejection_sampling_zero_residual(tv, dtype):
    # the hand-built case of the oracle's pin: a rejection whose residual
    # max(0, p - q) is exactly 0 (float32 as well) continues with the
    # target softmax, on the GPU as in the oracle
    import test_oracle_sampling as tos
    from oracle import sampling as osm
    pl, ql = tos.zero_residual_case()
    conv = (lambda x: synth.bf16_bits(x.astype(np.float32))) if dtype == "bf16" else (lambda x: x.astype(np.float32))
    for parent, tok, u in (([-1, 0], [0, 1], [0.0, 0.5]), ([-1, 0, 0], [0, 1, 0], [0.0, 0.5, 0.999])):
        n = len(parent)
        par, tk = np.array(parent, np.int32), np.array(tok, np.int32)
        un = np.array(u, np.float32)
        for uf in (0.001, 0.3, 0.999):
            ufa = np.array([uf], np.float32)
            off = np.array([0, n], np.int32)
            acc, best, path, bonus = tv.accept_rejection_sampling(dev(par), dev(tk), dev(conv(pl[:n])),
                                                                  dev(conv(ql[:n])), dev(off), dev(un), dev(ufa),
                                                                  max_depth=n - 1)
            sync()
            racc, rbest, rpath, rbonus, _, _ = osm.rejection_verify(par, tk, conv(pl[:n]), conv(ql[:n]), off, un,
                                                                    ufa, n - 1)
            assert host(acc)[0] == racc[0] and host(best)[0] == rbest[0] and host(bonus)[0] == rbonus[0]
            assert np.array_equal(host(path), rpath)
            assert rbonus[0] == (0 if n == 2 else 2)
