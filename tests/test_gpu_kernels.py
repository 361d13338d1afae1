"""GPU parity: each CUDA entry point against the CPU oracle on seeded inputs.

Integer outputs (argmax, top-k, depth/pos/masks, acceptance, table rows,
retrieval, selection) must match bit for bit; softmax quantities within 1e-5
relative; attention within max|delta| <= 1e-2 * max|ref| (bf16 inputs, fp32
accumulation) or 1e-4 * max|ref| (fp32 inputs).
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import attn_close, dev, host, out_to_f64
from oracle import accept as oacc
from oracle import alpha as oal
from oracle import attention as oatt
from oracle import dcut as odc
from oracle import graft as ogr
from oracle import mlp as omlp
from oracle import tree as otree
from oracle import vocab as ovoc

pytestmark = pytest.mark.gpu

ALPHA_RTOL = 1e-5
LSE_ATOL = 1e-5        # |delta lse| <= 1e-5  <=>  softmax mass within ~1e-5 relative
ATTN_BF16 = 1e-2
ATTN_F32 = 1e-4


@pytest.fixture(scope="module")
def tv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_tree_02_gb300 as m
    m.load_library()
    return m


def sync():
    torch.cuda.synchronize()


# ------------------------------------------------------------------ tree prep
def random_forest(rng, n, max_depth, p_root):
    parent = np.full(n, -1, np.int32)
    depth = np.zeros(n, np.int32)
    for i in range(1, n):
        if rng.random() < p_root:
            continue
        ok = np.nonzero(depth[:i] < max_depth)[0]
        p = int(ok[rng.integers(ok.size)])
        parent[i], depth[i] = p, depth[p] + 1
    return parent


@pytest.mark.parametrize("sizes,p_root", [([60], 0.0), ([1], 0.0), ([113] * 8, 0.0), ([16] * 64, 0.0),
                                          ([1024], 0.05), ([200, 1, 64, 65], 0.2)])
def test_tree_prep(tv, sizes, p_root):
    rng = np.random.default_rng(len(sizes) * 7 + sizes[0])
    parent = np.concatenate([random_forest(rng, n, 40, p_root) for n in sizes])
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    plen = rng.integers(0, 5000, len(sizes)).astype(np.int32)
    vis = rng.integers(0, 6000, parent.size).astype(np.int32) if p_root else None
    max_nodes = max(sizes)
    W = (max_nodes + 63) // 64
    d, pos, anc, v, err = tv.tv_tree_prep(dev(parent), dev(off), dev(plen), dev(vis), max_nodes, W)
    sync()
    vis_c = None if vis is None else np.minimum(vis, np.repeat(plen, sizes))
    rd, rpos, ranc, rvis = otree.tree_prep(parent, off, plen, vis_c, anc_words=W)
    assert np.array_equal(host(d), rd)
    assert np.array_equal(host(pos), rpos)
    assert np.array_equal(host(anc).view(np.uint64), ranc)
    assert np.array_equal(host(v), rvis)
    assert host(err)[0] == 0


def test_tree_prep_chain_max_nodes(tv):
    n = 1024
    parent = np.arange(-1, n - 1, dtype=np.int32)
    d, pos, anc, v, err = tv.tv_tree_prep(dev(parent), dev(np.array([0, n], np.int32)),
                                          dev(np.array([7], np.int32)), None, n, 16)
    sync()
    assert np.array_equal(host(d), np.arange(n))
    a = host(anc).view(np.uint64)
    for i in (0, 63, 64, 500, 1023):
        bits = [(int(a[i, j // 64]) >> (j % 64)) & 1 for j in range(n)]
        assert bits == [1] * (i + 1) + [0] * (n - i - 1)


# ---------------------------------------------------------------------- vocab
def check_vocab(tv, logits_np, k, row_idx=None, lse=True):
    R = logits_np.shape[0]
    rows = None if row_idx is None else row_idx
    am, ti, tvl, rm, rl = tv.vocab_argmax_topk(dev(logits_np), k=k, row_idx=dev(row_idx), out_rows=R,
                                               want_lse=lse)
    sync()
    sel = np.arange(R) if row_idx is None else row_idx
    ram, rti, rtv, rrm, rrl = ovoc.argmax_topk(logits_np, max(k, 1), rows=sel)
    assert np.array_equal(host(am)[sel], ram)
    if k:
        assert np.array_equal(host(ti)[sel], rti[:, :k])
        assert np.array_equal(host(tvl)[sel], rtv[:, :k])
    assert np.array_equal(host(rm)[sel], rrm)
    if lse:
        assert np.abs(host(rl)[sel].astype(np.float64) - rrl).max() <= LSE_ATOL
    return am


def test_vocab_tiny_fp32(tv):
    d = synth.tiny_tree()
    am = check_vocab(tv, d["logits"], 8)
    assert np.array_equal(host(am), d["planted"])


@pytest.mark.parametrize("k", [0, 1, 8, 16])
def test_vocab_bf16_graft_rows(tv, k):
    rng = synth.make_rng(90, k)
    planted = rng.integers(0, synth.QWEN3_VOCAB, 61).astype(np.int32)
    logits = synth.logits_rows(rng, 61, synth.QWEN3_VOCAB, 2.0, planted, "bf16")
    check_vocab(tv, logits, k)


def test_vocab_heavy_ties_bf16(tv):
    # integer-valued logits in a tiny range: thousands of exact ties per row
    rng = np.random.default_rng(3)
    x = rng.integers(-4, 5, (9, 20000)).astype(np.float32)
    check_vocab(tv, synth.bf16_bits(x), 16)
    check_vocab(tv, synth.bf16_bits(x), 8)


def test_vocab_all_equal_rows_use_fallback(tv):
    x = np.zeros((3, 9000), np.float32)
    check_vocab(tv, synth.bf16_bits(x), 8)
    check_vocab(tv, x, 16)


@pytest.mark.parametrize("V", [1001, 8193, 12345])
def test_vocab_ragged_width_and_stride(tv, V):
    rng = np.random.default_rng(V)
    x = (rng.standard_normal((5, V)) * 2).astype(np.float32)
    check_vocab(tv, x, 8)
    check_vocab(tv, synth.bf16_bits(x), 8)


def test_vocab_row_gather(tv):
    d = synth.dcut_batch(B=6, V=30000, with_attention=False)
    idx = np.array([0, 1, 2, 17, 18, 40, 95, 64], np.int32)
    check_vocab(tv, d["logits"], 8, row_idx=idx)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_vocab_host_resident_rows(tv, dtype):
    # logits in pinned host memory, read in place: only the gathered rows
    # are touched; results equal the oracle's (and so the device-resident call's)
    import torch
    d = synth.dcut_batch(B=8, V=synth.QWEN3_VOCAB, with_attention=False)
    x = d["logits"] if dtype == "bf16" else synth.bf16_to_f32(d["logits"])
    R = x.shape[0]
    idx = np.array([1, 3, 4, 17, 40, 77, 100, 127], np.int32)
    xt = torch.from_numpy(x.view(np.int16) if x.dtype == np.uint16 else x).pin_memory()
    am, ti, tvl, rm, rl = tv.vocab_argmax_topk(xt, k=8, row_idx=dev(idx), out_rows=R)
    sync()
    ram, rti, rtv, rrm, rrl = ovoc.argmax_topk(x, 8, rows=idx)
    assert np.array_equal(host(am)[idx], ram)
    assert np.array_equal(host(ti)[idx], rti)
    assert np.array_equal(host(tvl)[idx], rtv)
    assert np.array_equal(host(rm)[idx], rrm)
    assert np.abs(host(rl)[idx].astype(np.float64) - rrl).max() <= LSE_ATOL


def test_vocab_full_size_every_row(tv):
    # the D-cut workload at rho = 1: 1024 rows x 151936, every output compared
    d = synth.dcut_batch(with_attention=False)
    L = dev(d["logits"])
    am, ti, tvl, rm, rl = tv.vocab_argmax_topk(L, k=8)
    sync()
    assert np.array_equal(host(am), d["planted"])
    ram, rti, rtv, rrm, rrl = ovoc.argmax_topk(d["logits"], 8)
    assert np.array_equal(host(am), ram)
    assert np.array_equal(host(ti), rti)
    assert np.array_equal(host(tvl), rtv)
    assert np.array_equal(host(rm), rrm)
    assert np.abs(host(rl) - rrl).max() <= LSE_ATOL


# ---------------------------------------------------------------------- alpha
def check_alpha(tv, d, rows=None):
    a, pre, pm = tv.tree_tv_alpha(dev(d["lp"]), dev(d["lq"]), dev(d["branch_off"]), dev(d["mass_tok"]))
    sync()
    ra, _, rpre, rpm = oal.tv_alpha(d["lp"], d["lq"], d["branch_off"], d["mass_tok"], rows=rows)
    sel = np.arange(len(ra)) if rows is None else np.array(rows)
    np.testing.assert_allclose(host(a)[sel], ra[sel], rtol=ALPHA_RTOL)
    np.testing.assert_allclose(host(pm)[sel], rpm[sel], rtol=ALPHA_RTOL)
    if rows is None:
        np.testing.assert_allclose(host(pre), rpre, rtol=ALPHA_RTOL)
    return host(a), host(pre)


def test_alpha_small_forest(tv):
    d = synth.specopd_tree(prompt=32, response=96, n_anchor=6, W=5, V=20000, with_attention=False)
    check_alpha(tv, d)


@pytest.mark.parametrize("V", [40, 1001, 4104])
def test_alpha_small_and_ragged_vocab(tv, V):
    # V = 40: five of the eight slices of the one-read path are empty;
    # V = 1001: rows not a multiple of 8 elements take the two-pass path
    d = synth.specopd_tree(prompt=16, response=48, n_anchor=4, W=3, V=V, with_attention=False)
    check_alpha(tv, d)


def test_alpha_identity_is_one(tv):
    d = synth.specopd_tree(prompt=8, response=24, n_anchor=3, W=4, V=151936, with_attention=False)
    d["lq"] = d["lp"].copy()
    a, pre = check_alpha(tv, d)
    np.testing.assert_allclose(a, 1.0, rtol=ALPHA_RTOL)


def test_alpha_full_size_every_row(tv):
    # the SpecOPD scoring shape: 1024 rows x 151936, p and q; every row's
    # alpha and softmax mass, and every branch's running product
    from oracle_pool import OraclePool, alpha_task, split
    d = synth.specopd_tree(with_attention=False)
    a, pre, pm = tv.tree_tv_alpha(dev(d["lp"]), dev(d["lq"]), dev(d["branch_off"]), dev(d["mass_tok"]))
    sync()
    ra = np.full(1024, np.nan)
    rpm = np.full(1024, np.nan)
    with OraclePool({"lp": d["lp"], "lq": d["lq"], "mass_tok": d["mass_tok"]}) as pool:
        for rows, a_r, pm_r in pool.map(alpha_task, split(range(1024), 64)):
            ra[rows], rpm[rows] = a_r, pm_r
    np.testing.assert_allclose(host(a), ra, rtol=ALPHA_RTOL)
    np.testing.assert_allclose(host(pm), rpm, rtol=ALPHA_RTOL)
    np.testing.assert_allclose(host(pre), oal.branch_prefix(ra, d["branch_off"]), rtol=ALPHA_RTOL)
    assert np.all(np.diff(host(pre).reshape(64, 16), axis=1) <= 0)


# ----------------------------------------------------------------- acceptance
def check_accept(tv, parent, tok, argmax, off, valid=None, max_depth=None):
    sizes = np.diff(off)
    max_nodes = int(sizes.max())
    md = max_nodes - 1 if max_depth is None else max_depth
    al, best, path, bonus, pacc = tv.accept_longest_path(dev(parent), dev(tok), dev(argmax), dev(off),
                                                         dev(valid), max_nodes, md)
    sync()
    ral, rbest, rpath, rbonus, rpacc = oacc.accept_longest_path(parent, tok, argmax, off, valid, md)
    assert np.array_equal(host(al), ral)
    assert np.array_equal(host(best), rbest)
    assert np.array_equal(host(bonus), rbonus)
    assert np.array_equal(host(path), rpath)
    assert np.array_equal(host(pacc), rpacc)


@pytest.mark.parametrize("seed", range(6))
def test_accept_random_forests(tv, seed):
    rng = np.random.default_rng(seed)
    sizes = rng.integers(1, 200, 7)
    parent = np.concatenate([random_forest(rng, int(n), 12, 0.05 * (seed % 3)) for n in sizes])
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    V = 3
    tok = rng.integers(0, V, parent.size).astype(np.int32)
    argmax = rng.integers(0, V, parent.size).astype(np.int32)
    valid = (rng.random(parent.size) < 0.9).astype(np.uint8) if seed % 2 else None
    check_accept(tv, parent, tok, argmax, off, valid)


def test_accept_workloads(tv):
    d = synth.tiny_tree()
    check_accept(tv, d["parent"], d["tok"], d["planted"], d["node_off"])
    d = synth.dcut_batch(with_attention=False, with_logits=False)
    check_accept(tv, d["parent"], d["tok"], d["planted"], d["node_off"])
    d = synth.blockpilot_sweep(with_attention=False, with_mlp=False, V=1000)
    check_accept(tv, d["parent"], d["tok"], d["planted"], d["node_off"], max_depth=19)


def test_accept_chain_1024_and_truncated_path(tv):
    n = 1024
    parent = np.arange(-1, n - 1, dtype=np.int32)
    argmax = np.arange(n, dtype=np.int32)
    tok = np.concatenate([[5], np.arange(n - 1)]).astype(np.int32)
    tok[900] = -7
    check_accept(tv, parent, tok, argmax, np.array([0, n], np.int32))
    check_accept(tv, parent, tok, argmax, np.array([0, n], np.int32), max_depth=10)


# ------------------------------------------------------------------ Graft table
@pytest.mark.parametrize("n", [3000, 5000])   # ordered scan / last-index table
def test_adj_update_duplicates_invalid_and_bad_tokens(tv, n):
    rng = np.random.default_rng(1)
    V, k = 3000, 8
    adj = rng.integers(0, V, (V, k)).astype(np.int32)
    tok = rng.integers(0, 400, n).astype(np.int32)        # many duplicates
    tok[::97] = V + 3                                       # out of range
    tok[5::101] = -2
    topk = rng.integers(0, V, (n, k)).astype(np.int32)
    valid = (rng.random(n) < 0.8).astype(np.uint8)
    g = dev(adj)
    nb = tv.graft_adj_update(g, dev(tok), dev(topk), dev(valid))
    sync()
    ref = adj.copy()
    ok = valid.astype(bool) & (tok >= 0) & (tok < V)
    ogr.adj_update(ref, np.where(ok, tok, 0), topk, ok)
    assert np.array_equal(host(g), ref)
    assert host(nb)[0] == int((valid.astype(bool) & ~((tok >= 0) & (tok < V))).sum())


def test_adj_update_bulk_full_table(tv):
    rng = np.random.default_rng(2)
    V, k = synth.QWEN3_VOCAB, 8
    adj = rng.integers(0, V, (V, k)).astype(np.int32)
    tok = rng.permutation(V).astype(np.int32)
    tok[rng.choice(V, V // 3, replace=False)] = rng.integers(0, V, V // 3)   # duplicates everywhere
    topk = rng.integers(0, V, (V, k)).astype(np.int32)
    g = dev(adj)
    tv.graft_adj_update(g, dev(tok), dev(topk))
    sync()
    ref = adj.copy()
    last = {}
    for i, t in enumerate(tok):
        last[int(t)] = i
    idx = np.array(list(last.keys()))
    ref[idx] = topk[np.array(list(last.values()))]
    assert np.array_equal(host(g), ref)


def test_retrieve_matches_oracle(tv):
    tp, tr, off = tv.stage_templates()
    rng = np.random.default_rng(4)
    V, k, B = 1000, 8, 37
    adj = rng.integers(0, V, (V, k)).astype(np.int32)
    root = rng.integers(0, V, B).astype(np.int32)
    stage = rng.integers(0, 4, B).astype(np.int32)
    rtok, rpar, ns, err = tv.graft_retrieve(dev(adj), dev(root), dev(stage), dev(tp), dev(tr), dev(off), 52)
    sync()
    otp, otr, ooff = ogr.stage_templates()
    ertok, erpar, ens = ogr.retrieve(adj, root, stage, otp, otr, ooff, 52)
    assert np.array_equal(host(rtok), ertok)
    assert np.array_equal(host(rpar), erpar)
    assert np.array_equal(host(ns), ens)
    assert host(err)[0] == 0


def test_retrieve_bad_table_entry_flags_error(tv):
    tp, tr, off = tv.stage_templates()
    V, k = 50, 8
    adj = np.array([[(t + r + 1) % V for r in range(k)] for t in range(V)], np.int32)
    adj[3, 0] = V + 9                                        # poisoned successor
    rtok, rpar, ns, err = tv.graft_retrieve(dev(adj), dev(np.array([2], np.int32)),
                                            dev(np.array([0], np.int32)), dev(tp), dev(tr), dev(off), 52)
    sync()
    assert host(err)[0] == 1
    r = host(rtok)[0]
    # slot 0 = adj[2][0] = 3 is fine; slot 1 = adj[3][0] is poisoned, and so is its subtree
    assert r[0] == 3 and r[1] == -1 and r[2] == -1


# ---------------------------------------------------------------------- D-cut
@pytest.mark.parametrize("which", ["workload", "ties", "tiny", "t1500", "t4000", "t8192", "d0",
                                   "rho8", "nonmonotone", "zeros", "t1005"])
def test_dcut_select(tv, which):
    rng = np.random.default_rng(len(which))
    beta = lambda b, d: rng.beta(4.0, 1.5, (b, d)).astype(np.float32)
    rhos = list(synth.DCUT_RHOS)
    if which == "workload":
        conf = synth.dcut_batch(with_attention=False, with_logits=False)["conf"]
    elif which == "t1500":     # two keys per thread in the sorting network
        conf = beta(100, 14)
    elif which == "t4000":     # four keys per thread
        conf = beta(200, 19)
    elif which == "t8192":     # the largest batch the kernel takes
        conf = beta(512, 15)
    elif which == "d0":        # root-only requests: every score is 1, order = position
        conf = np.zeros((5000, 0), np.float32)
        rhos = [0.0, 0.3, 0.5001, 1.0]
    elif which == "rho8":      # the most budgets one call takes
        conf = beta(37, 20)
        rhos = [0.0, 0.01, 0.1, 0.25, 0.5, 0.75, 0.99, 1.0]
    elif which == "nonmonotone":   # confidences above 1: kept sets are not prefixes
        conf = rng.uniform(0.0, 2.0, (125, 15)).astype(np.float32)
        rhos = [0.2, 0.5, 0.8]
    elif which == "zeros":     # exact zero scores (their score word is all ones)
        conf = np.where(rng.random((60, 12)) < 0.2, 0.0, beta(60, 12)).astype(np.float32)
        rhos = [0.1, 0.5, 0.9, 1.0]
    elif which == "t1005":     # ragged: positions per cluster CTA not a multiple of 4
        conf = beta(67, 14)
    elif which == "ties":
        rng = np.random.default_rng(5)
        conf = rng.choice(np.array([1.0, 0.5, 0.25, 0.75], np.float32), (40, 9))
        rhos = [0.1, 0.33, 0.5, 0.77, 1.0]
    else:
        conf = np.array([[0.9, 0.2], [0.5, 0.5]], np.float32)
        rhos = [0.0, 0.2, 1.0]
    s, keep, kl, po, pi = tv.dcut_select(dev(conf), rhos)
    sync()
    rs, rkeep, rkl, rpo, rpi = odc.select(conf, rhos)
    assert np.array_equal(host(s), rs)                     # bit-exact fp32 products
    assert np.array_equal(host(keep), rkeep)
    assert np.array_equal(host(kl), rkl)
    assert np.array_equal(host(po), rpo)
    assert np.array_equal(host(pi), rpi)


def test_dcut_select_sorting_network_in_subprocess(tv):
    """Up to 2048 positions run on the cluster kernel; the single-CTA sorting
    network for the same sizes is checked in a process with TV_DCUT_PATH=sort."""
    import os
    import subprocess
    import sys
    code = (
        "import sys; sys.path.insert(0, 'tests'); sys.path.insert(0, '.');"
        "import test_gpu_kernels as t, speculative_decoding_tree_02_gb300 as tv;"
        "[t.test_dcut_select(tv, w) for w in ('workload', 'ties', 'tiny', 't1500', 'rho8', 'nonmonotone')];"
        "print('sort ok')")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, TV_DCUT_PATH="sort")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "sort ok" in r.stdout, r.stderr[-3000:]


# ------------------------------------------------------------------ attention
def run_attn(tv, d, nodes=None, node_cnt=None, rel=None):
    off, pre_off = d["node_off"], d["pre_off"]
    sizes = np.diff(off)
    max_nodes = int(sizes.max())
    max_prefix = int(np.diff(pre_off).max())
    plen = np.diff(pre_off).astype(np.int32)
    W = (max_nodes + 63) // 64
    _, _, anc, _, _ = tv.tv_tree_prep(dev(d["parent"]), dev(off), dev(plen), dev(d["vis_prefix"]),
                                      max_nodes, W)
    o, lse = tv.tree_verify_attn(dev(d["q"]), dev(d["k_pre"]), dev(d["v_pre"]), dev(pre_off),
                                 dev(d["k_tree"]), dev(d["v_tree"]), dev(off), anc, max_nodes, max_prefix,
                                 vis_prefix=dev(d["vis_prefix"]), node_cnt=dev(node_cnt))
    sync()
    ro, rlse = oatt.tree_attention(d["q"], d["k_pre"], d["v_pre"], pre_off, d["k_tree"], d["v_tree"], off,
                                   d["parent"], d["vis_prefix"], node_cnt=node_cnt, nodes=nodes)
    got = out_to_f64(o)
    if rel is None:
        rel = ATTN_BF16 if d["dtype"] == "bf16" else ATTN_F32
    ok, err, scale = attn_close(got, ro, rel)
    assert ok, (err, scale)
    m = ~np.isnan(rlse)
    assert np.abs(host(lse)[m] - rlse[m]).max() <= 1e-4
    return got, host(lse)


def test_attn_tiny_fp32(tv):
    run_attn(tv, synth.tiny_tree())


def test_attn_graft_shape_bf16(tv):
    st = synth.graft_static(V=1000)
    d = synth.graft_step(0, st)
    tp, tr, off = tv.stage_templates()
    nd = d["n_draft"]
    parent = tv.assemble_hybrid(d["parent_draft"], tp[off[d["stage"]]:off[d["stage"] + 1]])
    assert parent.size == d["N"]
    d["parent"] = parent
    run_attn(tv, d)


def test_attn_dcut_small_with_node_cnt(tv):
    d = synth.dcut_batch(B=6, P_min=1, P_max=700, V=64)
    cnt = np.array([16, 1, 5, 16, 9, 3], np.int32)
    run_attn(tv, d, node_cnt=cnt)


def run_attn_full(tv, d, node_cnt=None):
    """Every output of a full-size workload against the oracle."""
    off, pre_off = d["node_off"], d["pre_off"]
    sizes = np.diff(off)
    max_nodes, max_prefix = int(sizes.max()), int(np.diff(pre_off).max())
    plen = np.diff(pre_off).astype(np.int32)
    _, _, anc, _, _ = tv.tv_tree_prep(dev(d["parent"]), dev(off), dev(plen), dev(d["vis_prefix"]), max_nodes,
                                      (max_nodes + 63) // 64)
    o, lse = tv.tree_verify_attn(dev(d["q"]), dev(d["k_pre"]), dev(d["v_pre"]), dev(pre_off), dev(d["k_tree"]),
                                 dev(d["v_tree"]), dev(off), anc, max_nodes, max_prefix,
                                 vis_prefix=dev(d["vis_prefix"]), node_cnt=dev(node_cnt))
    sync()
    from oracle_pool import oracle_attention_all
    ro, rlse = oracle_attention_all(d, node_cnt)
    got = out_to_f64(o)
    ok, err, scale = attn_close(got, ro, ATTN_BF16)
    assert ok, (err, scale)
    m = ~np.isnan(rlse)
    assert np.abs(host(lse)[m] - rlse[m]).max() <= 1e-4
    return got, ro


def test_attn_dcut_full_size_every_node(tv):
    # 64 requests x 16 nodes, prefixes 512..4096: every node and head
    run_attn_full(tv, synth.dcut_batch(with_logits=False))


def test_attn_blockpilot_full_size_every_node(tv):
    # 8 requests x 113 nodes over 8192-token prefixes (the 64-row / 128-row
    # tensor-core tiles and their ragged last tile)
    run_attn_full(tv, synth.blockpilot_sweep(with_mlp=False, V=64))


def test_attn_specopd_full_size_every_node(tv):
    # 1024 branch nodes over one 4096-token trunk: all 32 128-row tiles
    run_attn_full(tv, synth.specopd_tree(with_logits=False))


def test_attn_edge_cases(tv):
    # empty prefix, single node, d = 64 bf16, one query head per KV head
    rng = synth.make_rng(77)
    for (P, n, Hq, Hkv, d_, dt) in [(0, 1, 4, 4, 64, "bf16"), (0, 9, 8, 2, 128, "f32"),
                                    (33, 70, 2, 2, 64, "bf16"), (5, 3, 16, 1, 128, "bf16")]:
        parent = synth.random_tree(rng, n, 6)
        att = synth.attention_tensors(rng, n, P, Hq, Hkv, d_, dt)
        dd = dict(parent=parent, node_off=np.array([0, n], np.int32), pre_off=np.array([0, P], np.int32),
                  vis_prefix=None, dtype=dt, **att)
        run_attn(tv, dd)


def test_attn_zero_visible_prefix(tv):
    d = synth.specopd_tree(prompt=4, response=60, n_anchor=5, W=3, V=64, Hq=4, Hkv=2, d=64)
    d["vis_prefix"] = d["vis_prefix"].copy()
    d["vis_prefix"][:3] = 0
    run_attn(tv, d)


# ----------------------------------------------------------------- BlockPilot
def test_blockpilot_mlp_full_size(tv):
    d = synth.blockpilot_sweep(with_attention=False)
    L = dev(d["last_logits"])
    _, _, _, _, lse = tv.vocab_argmax_topk(L, k=0)
    z, choice, bsize = tv.blockpilot_mlp(L, lse, dev(d["W1"]), dev(d["W2"]), block=d["block"])
    sync()
    rz, rchoice, rbsize = omlp.blockpilot(d["last_logits"], d["W1"], d["b1"], d["W2"], d["b2"], d["block"])
    zg = host(z).astype(np.float64)
    tol = 1e-4 * np.abs(rz).max()
    assert np.abs(zg - rz).max() <= tol
    for r in range(len(rchoice)):
        srt = np.sort(rz[r])[::-1]
        if srt[0] - srt[1] > 2 * tol:                         # decision fixed by the oracle's margin
            assert host(choice)[r] == rchoice[r]
            assert host(bsize)[r] == rbsize[r]
        else:                                                  # near-tie: must pick one of the tied
            assert rz[r, host(choice)[r]] >= srt[0] - 2 * tol
    assert set(host(bsize).tolist()) <= set(d["sizes"].tolist())


def test_blockpilot_zero_weights(tv):
    rng = np.random.default_rng(0)
    V, H, C = 3000, 256, 7
    logits = synth.bf16_bits(rng.standard_normal((3, V)).astype(np.float32))
    L = dev(logits)
    _, _, _, _, lse = tv.vocab_argmax_topk(L, k=0)
    W1 = dev(np.zeros((V, H), np.uint16))
    W2 = dev(np.zeros((H, C), np.uint16))
    z, choice, bsize = tv.blockpilot_mlp(L, lse, W1, W2, block=16)
    sync()
    assert np.all(host(z) == 0) and np.all(host(choice) == 0) and np.all(host(bsize) == 13)


@pytest.mark.parametrize("B,V,H,C", [(5, 20011, 512, 7), (1, 4099, 256, 32), (8, 150, 256, 3), (12, 3001, 256, 7)])
def test_blockpilot_mlp_biases_and_workspace_reuse(tv, B, V, H, C):
    """Biases, ragged request counts, few hidden tiles (many K splits each), a
    workspace that starts dirty and is reused: the split-K arrival counters
    must be cleared by the call and leave no state behind.  B = 12 runs the
    CUDA-core fallback."""
    rng = np.random.default_rng(B * 1000 + H)
    logits = synth.bf16_bits((3.0 * rng.standard_normal((B, V))).astype(np.float32))
    W1 = synth.bf16_bits((0.05 * rng.standard_normal((V, H))).astype(np.float32))
    W2 = synth.bf16_bits((0.05 * rng.standard_normal((H, C))).astype(np.float32))
    b1 = (0.01 * rng.standard_normal(H)).astype(np.float32)
    b2 = (0.01 * rng.standard_normal(C)).astype(np.float32)
    L = dev(logits)
    _, _, _, _, lse = tv.vocab_argmax_topk(L, k=0)
    need = tv.load_library().blockpilot_mlp_workspace_size(B, V, H)
    ws = torch.full((need,), 0xA5, dtype=torch.uint8, device="cuda")
    rz, rchoice, _ = omlp.blockpilot(logits, W1, b1, W2, b2, 16)
    tol = 1e-4 * np.abs(rz).max() + 1e-6
    for _ in range(3):
        z, choice, bsize = tv.blockpilot_mlp(L, lse, dev(W1), dev(W2), b1=dev(b1), b2=dev(b2), block=16, ws=ws)
        sync()
        zg = host(z).astype(np.float64)
        assert np.abs(zg - rz).max() <= tol
        for r in range(B):
            srt = np.sort(rz[r])[::-1]
            if C == 1 or srt[0] - srt[1] > 2 * tol:
                assert host(choice)[r] == rchoice[r]
            assert host(bsize)[r] == 16 - (C - 1) // 2 + host(choice)[r]


def test_attn_simt_path_on_bf16_in_subprocess(tv):
    """bf16 / head_dim 128 normally runs on the tensor cores; the SIMT kernel
    for the same shapes is checked in a process with TV_ATTN_PATH=simt."""
    import os
    import subprocess
    import sys
    code = (
        "import sys; sys.path.insert(0, 'tests'); sys.path.insert(0, '.');"
        "import test_gpu_kernels as t, synth, speculative_decoding_tree_02_gb300 as tv;"
        "t.run_attn(tv, synth.dcut_batch(B=6, P_min=1, P_max=700, V=64),"
        " node_cnt=__import__('numpy').array([16, 1, 5, 16, 9, 3], 'int32'));"
        "st = synth.graft_static(V=1000); d = synth.graft_step(3, st); tp, tr, off = tv.stage_templates();"
        "d['parent'] = tv.assemble_hybrid(d['parent_draft'], tp[off[d['stage']]:off[d['stage'] + 1]]);"
        "t.run_attn(tv, d); print('simt ok')")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, TV_ATTN_PATH="simt")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "simt ok" in r.stdout, r.stderr[-3000:]


def test_attn_status_word_clear(tv):
    """The tensor-core kernel reports no pipeline timeout on a normal call."""
    d = synth.dcut_batch(B=4, P_min=100, P_max=900, V=64)
    off, pre_off = d["node_off"], d["pre_off"]
    plen = np.diff(pre_off).astype(np.int32)
    _, _, anc, _, _ = tv.tv_tree_prep(dev(d["parent"]), dev(off), dev(plen), None, 16, 1)
    need = tv.load_library().tree_verify_attn_workspace_size(4, 16, int(plen.max()), 32, 8, 128, 1)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    ws[:4] = 7
    tv.tree_verify_attn(dev(d["q"]), dev(d["k_pre"]), dev(d["v_pre"]), dev(pre_off), dev(d["k_tree"]),
                        dev(d["v_tree"]), dev(off), anc, 16, int(plen.max()), ws=ws)
    sync()
    assert int(ws[:4].view(torch.int32).item()) == 0


def test_host_validation_with_real_buffers(tv):
    """The calls the host-side checks must refuse, given a real 64 MB device
    buffer for every array argument (large enough for any launch these
    argument lists could describe), so a validation regression could not
    reach memory outside it."""
    import ctypes
    import test_host_abi as tha
    buf = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
    for want, call in tha.validation_calls(tv.load_library(), ctypes.c_void_p(buf.data_ptr())):
        assert call() == want
    torch.cuda.synchronize()
    assert int(buf.count_nonzero()) == 0                  # nothing ran


def test_vocab_expired_wait_reports_failure_in_subprocess(tv):
    """When a bounded wait of the streaming kernels runs out, every reduced row
    reports failure (argmax -1, NaN values) and the workspace status word is
    nonzero, instead of a merge of stale chunk records.  The failure is planted
    on the host (TV_TEST_VOCAB_STATUS sets the status word where the call
    would clear it), so no wait actually runs out and nothing faults."""
    import os
    import subprocess
    import sys
    code = (
        "import sys; sys.path.insert(0, 'tests'); sys.path.insert(0, '.');"
        "import numpy as np, torch, synth, speculative_decoding_tree_02_gb300 as tv;"
        "x = synth.bf16_bits(np.random.default_rng(1).standard_normal((5, 40000)).astype(np.float32));"
        "L = torch.from_numpy(x.view(np.int16)).cuda();"
        "ws = torch.zeros(tv.load_library().vocab_argmax_topk_workspace_size(5, 40000, 8), dtype=torch.uint8,"
        " device='cuda');"
        "am, ti, tvl, rm, rl = tv.vocab_argmax_topk(L, k=8, ws=ws); torch.cuda.synchronize();"
        "assert (am == -1).all() and (ti == -1).all() and torch.isnan(tvl).all();"
        "assert torch.isnan(rm).all() and torch.isnan(rl).all();"
        "assert int(ws[:4].view(torch.int32).item()) == 3;"
        "o = (torch.zeros(5, dtype=torch.int32, device='cuda'), torch.zeros((5, 8), dtype=torch.int32, device='cuda'),"
        " torch.zeros((5, 8), device='cuda'), torch.zeros(5, device='cuda'), torch.zeros(5, device='cuda'));"
        "tv.vocab_argmax_topk_noalloc(L, *o, k=8); torch.cuda.synchronize();"
        "assert (o[0] == -1).all() and torch.isnan(o[4]).all();"
        "print('failure reported')")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, TV_TEST_VOCAB_STATUS="3")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "failure reported" in r.stdout, r.stderr[-3000:]


def test_vocab_status_word_clear_after_a_normal_call(tv):
    x = synth.bf16_bits(np.random.default_rng(2).standard_normal((5, 40000)).astype(np.float32))
    ws = torch.full((tv.load_library().vocab_argmax_topk_workspace_size(5, 40000, 8),), 7, dtype=torch.uint8,
                    device="cuda")
    am = tv.vocab_argmax_topk(dev(x), k=8, ws=ws)[0]
    sync()
    assert int(ws[:4].view(torch.int32).item()) == 0
    assert np.array_equal(host(am), ovoc.argmax_topk(x, 1)[0])



@pytest.mark.parametrize("seed", range(6))
def test_attn_random_forests_bf16(tv, seed):
    """Random request counts, tree sizes (one node to a few 128-row tiles),
    prefix lengths (zero to a few thousand keys), per-node visible prefixes or
    none, and node_cnt or none: whatever tile size, piece count and plan order
    the call takes, every verified output matches the oracle."""
    rng = synth.make_rng(63, seed)
    B = int(rng.integers(1, 6))
    sizes = [int(x) for x in rng.integers(1, 150, B)]
    parent = np.concatenate([synth.random_tree(rng, n, int(rng.integers(1, 12))) for n in sizes])
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    plen = rng.integers(0, 3000, B).astype(np.int32)
    vis = None
    if seed % 2:
        vis = np.concatenate([rng.integers(0, plen[r] + 1, sizes[r]) for r in range(B)]).astype(np.int32)
    cnt = np.array([int(rng.integers(1, n + 1)) for n in sizes], np.int32) if seed % 3 == 0 else None
    att = synth.attention_tensors(rng, int(off[-1]), max(1, int(plen.sum())), 32, 8, 128, "bf16")
    d = dict(parent=parent, node_off=off, pre_off=np.concatenate([[0], np.cumsum(plen)]).astype(np.int32),
             vis_prefix=vis, dtype="bf16", **att)
    run_attn(tv, d, node_cnt=cnt)


@pytest.mark.parametrize("sizes,cnt,P", [([70, 45, 130], [50, 45, 7], 900), ([160, 33], [129, 1], 2500)])
def test_attn_128_row_tiles_node_cnt_and_visible_prefixes(tv, sizes, cnt, P):
    """128-row tiles whose requests are cut short by node_cnt (only the first
    cnt nodes verified) and whose nodes see per-node prefixes: the planner's
    per-tile visible keys and node counts decide the pieces and their order."""
    rng = synth.make_rng(62, len(sizes) * 1000 + P)
    parent = np.concatenate([synth.random_tree(rng, n, 9) for n in sizes])
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    plen = rng.integers(P // 3, P + 1, len(sizes)).astype(np.int32)
    vis = np.concatenate([rng.integers(0, plen[r] + 1, sizes[r]) for r in range(len(sizes))]).astype(np.int32)
    att = synth.attention_tensors(rng, int(off[-1]), int(plen.sum()), 32, 8, 128, "bf16")
    d = dict(parent=parent, node_off=off, pre_off=np.concatenate([[0], np.cumsum(plen)]).astype(np.int32),
             vis_prefix=vis, dtype="bf16", **att)
    run_attn(tv, d, node_cnt=np.array(cnt, np.int32))


@pytest.mark.parametrize("sizes,P", [([80, 40, 1, 33], 700), ([96], 3000), ([200, 130], 257), ([61], 8192),
                                     ([29], 5000)])
def test_attn_128_row_tiles_ragged(tv, sizes, P):
    """128-row tiles with 128-key blocks: several tiles per request, ragged
    last tiles, a one-node request, and key pieces with their merge (few
    tiles over a long prefix: up to four 2048-key pieces, a ragged last one)."""
    rng = synth.make_rng(61, len(sizes) * 1000 + P)
    parent = np.concatenate([synth.random_tree(rng, n, 9) for n in sizes])
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    plen = rng.integers(P // 2, P + 1, len(sizes)).astype(np.int32)
    att = synth.attention_tensors(rng, int(off[-1]), int(plen.sum()), 32, 8, 128, "bf16")
    d = dict(parent=parent, node_off=off, pre_off=np.concatenate([[0], np.cumsum(plen)]).astype(np.int32),
             vis_prefix=None, dtype="bf16", **att)
    run_attn(tv, d)
