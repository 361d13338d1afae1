"""Tree-masked grouped-query attention over a shared KV prefix (fp64).

Definition followed (Graft page section 2, third gear; SpecOPD page section 02,
full-attention row of the architecture table and the proposal-tree stage of
the flow chart): every candidate node is scored in one forward pass, and node
i attends to the visible part of the shared prefix/trunk plus its own path
from the root — the same result as ordinary causal attention on the sequence
``prefix[:vis_i] ++ path(root -> i)`` taken at its last position.

The key list is built from ``parent`` by walking to the root, not from any
bitmask, so this routine is independent of the ancestor-mask step.

Heads: query head h reads KV head ``h // (Hq // Hkv)`` (grouped-query
attention with contiguous groups).  Logits are ``scale * q.k``; ``lse`` is the
natural-log log-sum-exp of those logits.
"""
from __future__ import annotations

import numpy as np

from .tree import path_to_root


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of raw bf16 patterns (uint16) to float64."""
    u = np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def as_f64(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return bf16_to_f64(x)
    return x.astype(np.float64)


def node_attention(q_i, keys, vals, scale):
    """One node, all heads.  q_i [Hq, d], keys/vals [L, Hkv, d] -> o [Hq, d], lse [Hq]."""
    Hq = q_i.shape[0]
    Hkv = keys.shape[1]
    g = Hq // Hkv
    o = np.empty_like(q_i)
    lse = np.empty(Hq)
    for h in range(Hq):
        kv = h // g
        s = (keys[:, kv, :] @ q_i[h]) * scale
        m = s.max()
        w = np.exp(s - m)
        l = w.sum()
        o[h] = (w @ vals[:, kv, :]) / l
        lse[h] = m + np.log(l)
    return o, lse


def tree_attention(q, k_pre, v_pre, pre_off, k_tree, v_tree, node_off, parent,
                   vis_prefix=None, scale=None, node_cnt=None, nodes=None):
    """Attention output and lse for every node (or only ``nodes``, a list of
    global node indices).  Unvisited rows are NaN.

    q [n, Hq, d]; k_pre/v_pre [sum P, Hkv, d] with request r's prefix at
    ``pre_off[r]:pre_off[r+1]``; k_tree/v_tree [n, Hkv, d] (node i's own
    key/value row); ``node_cnt[r]`` (optional) limits request r to its first
    node_cnt[r] nodes."""
    q = as_f64(q)
    n, Hq, d = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    node_off = np.asarray(node_off)
    pre_off = np.asarray(pre_off)
    out = np.full((n, Hq, d), np.nan)
    lse = np.full((n, Hq), np.nan)
    want = None if nodes is None else set(int(x) for x in nodes)
    kp_cache = {}
    for r in range(node_off.size - 1):
        n0, n1 = int(node_off[r]), int(node_off[r + 1])
        cnt = n1 - n0 if node_cnt is None else int(node_cnt[r])
        p0, p1 = int(pre_off[r]), int(pre_off[r + 1])
        for i in range(cnt):
            gi = n0 + i
            if want is not None and gi not in want:
                continue
            vp = (p1 - p0) if vis_prefix is None else int(vis_prefix[gi])
            key = (p0, vp)
            if key not in kp_cache:
                kp_cache.clear()
                kp_cache[key] = (as_f64(k_pre[p0:p0 + vp]), as_f64(v_pre[p0:p0 + vp]))
            kp, vpv = kp_cache[key]
            path = [n0 + j for j in path_to_root(parent, n0, i)]
            keys = np.concatenate([kp, as_f64(k_tree[path])], axis=0)
            vals = np.concatenate([vpv, as_f64(v_tree[path])], axis=0)
            out[gi], lse[gi] = node_attention(q[gi], keys, vals, scale)
    return out, lse
