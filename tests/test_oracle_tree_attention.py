"""Pins for the oracle's tree structure and tree-masked attention.

Each pin checks the oracle against something other than itself: the
transitive closure of the parent relation, torch's causal SDPA on chains
(a chain tree is ordinary decoding: BlockPilot page intro, SpecOPD page
section 01), a dense masked-softmax formulation, exact special cases, and the
locality property behind the Graft superset argument (Graft page section 3).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt
from oracle import tree as otree


def closure_ancestors(parent):
    """Reflexive-transitive closure of child->parent edges (Warshall)."""
    n = len(parent)
    A = np.eye(n, dtype=bool)
    for i, p in enumerate(parent):
        if p >= 0:
            A[i, p] = True
    for k in range(n):
        A |= A[:, [k]] & A[[k], :]
    return A


def random_forest(rng, n, max_depth, p_root=0.0):
    parent = np.full(n, -1, np.int32)
    depth = np.zeros(n, np.int32)
    for i in range(1, n):
        if rng.random() < p_root:
            continue
        ok = np.nonzero(depth[:i] < max_depth)[0]
        p = int(ok[rng.integers(ok.size)])
        parent[i], depth[i] = p, depth[p] + 1
    return parent


@pytest.mark.parametrize("seed", range(6))
def test_ancestor_mask_matches_closure(seed):
    rng = np.random.default_rng(seed)
    sizes = [1, 7, 64, 65, 130][: 2 + seed % 4]
    parents, off = [], [0]
    for n in sizes:
        parents.append(random_forest(rng, n, 12, p_root=0.1 if seed % 2 else 0.0))
        off.append(off[-1] + n)
    parent = np.concatenate(parents)
    plen = rng.integers(0, 50, len(sizes))
    depth, pos, anc, vis = otree.tree_prep(parent, np.array(off), plen)
    for r, n in enumerate(sizes):
        A = closure_ancestors(parents[r])
        for i in range(n):
            bits = [(int(anc[off[r] + i, j // 64]) >> (j % 64)) & 1 for j in range(n)]
            assert bits == A[i].astype(int).tolist()
            assert depth[off[r] + i] == A[i].sum() - 1
            assert vis[off[r] + i] == plen[r]
            assert pos[off[r] + i] == plen[r] + depth[off[r] + i]
        # bits beyond the request's nodes stay clear
        W = anc.shape[1]
        for i in range(n):
            for j in range(n, 64 * W):
                assert (int(anc[off[r] + i, j // 64]) >> (j % 64)) & 1 == 0


def test_chain_mask_is_lower_triangular():
    parent = np.arange(-1, 99, dtype=np.int32)
    _, pos, anc, _ = otree.tree_prep(parent, np.array([0, 100]), np.array([5]))
    for i in range(100):
        for j in range(100):
            assert ((int(anc[i, j // 64]) >> (j % 64)) & 1) == (1 if j <= i else 0)
    assert pos.tolist() == list(range(5, 105))


def sdpa_causal(q_seq, k_seq, v_seq, scale):
    """torch SDPA (CPU, float64) with repeat-interleaved KV heads.
    q_seq [L, Hq, d], k/v [L, Hkv, d] -> [L, Hq, d]."""
    g = q_seq.shape[1] // k_seq.shape[1]
    q = torch.from_numpy(q_seq).permute(1, 0, 2)[None]
    k = torch.from_numpy(k_seq).repeat_interleave(g, dim=1).permute(1, 0, 2)[None]
    v = torch.from_numpy(v_seq).repeat_interleave(g, dim=1).permute(1, 0, 2)[None]
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("Hq,Hkv,P,n", [(4, 1, 128, 16), (8, 2, 37, 9), (6, 3, 0, 5)])
def test_chain_equals_causal_sdpa(Hq, Hkv, P, n):
    rng = np.random.default_rng(Hq * 100 + P)
    d = 16
    parent = np.arange(-1, n - 1, dtype=np.int32)
    q = rng.standard_normal((n, Hq, d))
    kt, vt = rng.standard_normal((n, Hkv, d)), rng.standard_normal((n, Hkv, d))
    kp, vp = rng.standard_normal((P, Hkv, d)), rng.standard_normal((P, Hkv, d))
    scale = 1.0 / np.sqrt(d)
    o, lse = oatt.tree_attention(q, kp, vp, [0, P], kt, vt, [0, n], parent, scale=scale)
    q_seq = np.concatenate([np.zeros((P, Hq, d)), q])
    ref = sdpa_causal(q_seq, np.concatenate([kp, kt]), np.concatenate([vp, vt]), scale)[P:]
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)


def test_forest_with_visible_prefix_equals_per_branch_sdpa():
    """SpecOPD proposal forest: branch b sees trunk[:a_b+1] and its own earlier nodes."""
    d = synth.specopd_tree(prompt=16, response=48, n_anchor=5, W=4, V=64, Hq=4, Hkv=2, d=8)
    f = lambda x: oatt.as_f64(x)
    o, _ = oatt.tree_attention(d["q"], d["k_pre"], d["v_pre"], d["pre_off"], d["k_tree"],
                               d["v_tree"], d["node_off"], d["parent"], d["vis_prefix"])
    W = d["W"]
    for b, a in enumerate(d["anchors"]):
        sl = slice(b * W, (b + 1) * W)
        P = int(a) + 1
        q_seq = np.concatenate([np.zeros((P, 4, 8)), f(d["q"][sl])])
        ks = np.concatenate([f(d["k_pre"][:P]), f(d["k_tree"][sl])])
        vs = np.concatenate([f(d["v_pre"][:P]), f(d["v_tree"][sl])])
        ref = sdpa_causal(q_seq, ks, vs, 1.0 / np.sqrt(8))[P:]
        np.testing.assert_allclose(o[sl], ref, rtol=1e-12, atol=1e-12)


def dense_masked_attention(q, kp, vp, kt, vt, parent, scale, vis):
    """All keys (prefix ++ every tree node) with a 0/1 mask from the closure."""
    A = closure_ancestors(parent)
    n, Hq, d = q.shape
    Hkv = kt.shape[1]
    g = Hq // Hkv
    keys = np.concatenate([kp, kt])
    vals = np.concatenate([vp, vt])
    P = kp.shape[0]
    out = np.zeros_like(q)
    for i in range(n):
        mask = np.concatenate([np.arange(P) < vis[i], A[i]])
        for h in range(Hq):
            s = keys[:, h // g, :] @ q[i, h] * scale
            s = np.where(mask, s, -np.inf)
            w = np.exp(s - s.max())
            out[i, h] = (w / w.sum()) @ vals[:, h // g, :]
    return out


@pytest.mark.parametrize("seed", range(4))
def test_tree_equals_dense_masked_formulation(seed):
    rng = np.random.default_rng(seed)
    n, P, Hq, Hkv, d = 13, 11, 4, 2, 8
    parent = random_forest(rng, n, 4, p_root=0.15 * (seed % 2))
    vis = rng.integers(0, P + 1, n)
    q = rng.standard_normal((n, Hq, d))
    kt, vt = rng.standard_normal((n, Hkv, d)), rng.standard_normal((n, Hkv, d))
    kp, vp = rng.standard_normal((P, Hkv, d)), rng.standard_normal((P, Hkv, d))
    o, _ = oatt.tree_attention(q, kp, vp, [0, P], kt, vt, [0, n], parent, vis_prefix=vis, scale=0.3)
    ref = dense_masked_attention(q, kp, vp, kt, vt, parent, 0.3, vis)
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)


def test_single_visible_key_returns_its_value():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 4, 8))
    kt, vt = rng.standard_normal((1, 2, 8)), rng.standard_normal((1, 2, 8))
    empty = np.zeros((0, 2, 8))
    o, lse = oatt.tree_attention(q, empty, empty, [0, 0], kt, vt, [0, 1], np.array([-1]), scale=0.5)
    for h in range(4):
        assert np.array_equal(o[0, h], vt[0, h // 2])
        assert lse[0, h] == pytest.approx(0.5 * float(kt[0, h // 2] @ q[0, h]), abs=1e-15)


def test_locality_adding_nodes_leaves_existing_outputs_unchanged():
    """Graft superset argument: extra candidates never disturb existing ones."""
    d = synth.tiny_tree(N=40, P=20)
    args = (d["k_pre"], d["v_pre"], d["pre_off"])
    o_full, _ = oatt.tree_attention(d["q"], *args, d["k_tree"], d["v_tree"], d["node_off"], d["parent"])
    o_sub, _ = oatt.tree_attention(d["q"][:25], *args, d["k_tree"][:25], d["v_tree"][:25],
                                   [0, 25], d["parent"][:25])
    assert np.array_equal(o_full[:25], o_sub)


def test_non_ancestor_rows_do_not_matter():
    d = synth.tiny_tree(N=30, P=10)
    parent = d["parent"]
    A = closure_ancestors(parent)
    kt, vt = d["k_tree"].copy(), d["v_tree"].copy()
    i = 29
    others = [j for j in range(30) if not A[i, j]]
    assert others
    kt[others] += 7.0
    vt[others] -= 3.0
    args = (d["k_pre"], d["v_pre"], d["pre_off"])
    o1, _ = oatt.tree_attention(d["q"], *args, d["k_tree"], d["v_tree"], d["node_off"], parent, nodes=[i])
    o2, _ = oatt.tree_attention(d["q"], *args, kt, vt, d["node_off"], parent, nodes=[i])
    assert np.array_equal(o1[i], o2[i])


def test_bf16_widening_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x3F00, 0x0000, 0x4049], np.uint16)
    assert oatt.bf16_to_f64(bits).tolist() == [1.0, -2.0, 0.5, 0.0, 3.140625]


def test_large_logits_stay_finite_and_match_sdpa():
    """Logit spreads far beyond exp's range: the max-shifted softmax must hold."""
    rng = np.random.default_rng(11)
    n, P, Hq, Hkv, d = 6, 9, 4, 2, 8
    parent = np.arange(-1, n - 1, dtype=np.int32)
    q = rng.standard_normal((n, Hq, d)) * 400.0
    kt, vt = rng.standard_normal((n, Hkv, d)), rng.standard_normal((n, Hkv, d))
    kp, vp = rng.standard_normal((P, Hkv, d)), rng.standard_normal((P, Hkv, d))
    o, lse = oatt.tree_attention(q, kp, vp, [0, P], kt, vt, [0, n], parent, scale=1.0)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    q_seq = np.concatenate([np.zeros((P, Hq, d)), q])
    ref = sdpa_causal(q_seq, np.concatenate([kp, kt]), np.concatenate([vp, vt]), 1.0)[P:]
    np.testing.assert_allclose(o, ref, rtol=1e-9, atol=1e-9)
