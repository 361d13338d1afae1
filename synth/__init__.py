"""Seeded synthetic inputs for batched speculative-tree verification.

This module only *makes inputs*: random trees, tokens, logits, attention
tensors, draft confidences and weights, with the shapes and value
distributions of the five verification workloads.  It holds none of the
verification arithmetic (no masks, softmax, reductions, acceptance, table
updates or selection): those live in the CUDA library and, independently,
in the CPU oracle.  Both sides consume the arrays returned here.

Conventions
-----------
* Every generator draws from ``numpy.random.PCG64`` seeded with
  ``1000 * workload + step`` (``make_rng``).
* Integer arrays are ``int32``; bf16 tensors are returned as their raw 16-bit
  patterns (``uint16``), fp32 tensors as ``float32``.
* Tree arrays are flattened over requests: ``node_off[r]:node_off[r+1]`` are
  the nodes of request ``r`` and ``parent`` holds request-local indices, with
  ``-1`` for a root.  Parents always precede their children.
* Attention tensors are token-major: ``[tokens, heads, head_dim]``.

Workloads (sizes are the defaults; every generator takes smaller sizes for
tests, keeping the structure):

1. tiny tree verify: V=1000, prefix 128, one 60-node tree, 4/1 heads,
   head_dim 64, fp32 N(0,1); fp32 logits N(0,1) with a planted argmax; child
   token = parent's argmax with p=0.7; 1000x8 successor table.
2. Graft-shaped single request: V=151936 bf16 logits N(0, std 2) with a
   planted argmax; 32/8 heads, head_dim 128, prefix 2048; a 60-slot hybrid
   tree whose draft part has 8/24/40/60 nodes (pruning stage drawn
   uniformly) and whose retrieval part comes from the successor table.
3. D-cut batched block verify: 64 requests, each a chain of 1 bonus + 15
   drafts, prefix lengths uniform in [512, 4096], confidences Beta(4, 1.5),
   draft token = target argmax with probability equal to the confidence.
4. BlockPilot block-size sweep: 8 requests, prefix 8192, 32/8 heads, a root
   plus seven draft chains of 13..19 tokens (113 nodes); last-prefill logits
   and a 151936->2048->7 MLP with N(0, 0.02) bf16 weights.
5. SpecOPD proposal tree: 4096-token trunk (1024 prompt + 3072 response),
   64 distinct sorted anchors in the response, 16-token branch per anchor
   (1024 nodes), target and draft bf16 logits N(0, std 2).
"""
from __future__ import annotations

import numpy as np

QWEN3_VOCAB = 151936
DCUT_RHOS = (0.25, 0.5, 0.75, 1.0)
GRAFT_BUDGET = 60
# draft/retrieval split of the 60 verification slots for the pruning stages
# root, depth 1, depth 5 and "no pruning" (Graft page, section 2).
GRAFT_STAGE_DRAFT = (8, 24, 40, 60)


def make_rng(workload: int, step: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(1000 * workload + step))


# ---------------------------------------------------------------------------
# bf16 storage (data encoding only)
# ---------------------------------------------------------------------------
def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return the bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    out = np.empty(u.shape, np.uint16)
    # chunked to keep temporaries small for the 600 MB tensors
    flat_u, flat_o = u.reshape(-1), out.reshape(-1)
    step = 1 << 24
    for s in range(0, flat_u.size, step):
        c = flat_u[s:s + step]
        bias = ((c >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
        flat_o[s:s + step] = ((c + bias) >> np.uint32(16)).astype(np.uint16)
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return bf16_bits(x)


# ---------------------------------------------------------------------------
# building blocks
# ---------------------------------------------------------------------------
def random_tree(rng: np.random.Generator, n: int, max_depth: int) -> np.ndarray:
    """Parent array of an n-node tree rooted at node 0, depth <= max_depth.

    Node i picks its parent uniformly among the earlier nodes whose depth is
    below max_depth."""
    parent = np.full(n, -1, np.int32)
    depth = np.zeros(n, np.int32)
    for i in range(1, n):
        ok = np.nonzero(depth[:i] < max_depth)[0]
        p = int(ok[rng.integers(ok.size)])
        parent[i] = p
        depth[i] = depth[p] + 1
    return parent


def plant(rows_f32: np.ndarray, planted: np.ndarray, dtype: str) -> np.ndarray:
    """Give every row a unique maximum at ``planted[row]``.

    The row is drawn first; the planted entry is then set to the row maximum
    plus 1.0, rounded to the row's storage type (bf16 spacing below 32 is at
    most 0.125, so the planted value stays strictly above every other entry).
    Returns fp32 rows, or bf16 bits when ``dtype == 'bf16'``."""
    if dtype == "bf16":
        bits = bf16_bits(rows_f32)
        vals = bf16_to_f32(bits)
        top = vals.max(axis=1) + np.float32(1.0)
        bits[np.arange(bits.shape[0]), planted] = bf16_bits(top)
        return bits
    out = np.ascontiguousarray(rows_f32, np.float32).copy()
    out[np.arange(out.shape[0]), planted] = out.max(axis=1) + np.float32(1.0)
    return out


def logits_rows(rng: np.random.Generator, rows: int, V: int, std: float,
                planted: np.ndarray | None, dtype: str) -> np.ndarray:
    x = rng.standard_normal(size=(rows, V), dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if planted is None:
        return bf16_bits(x) if dtype == "bf16" else x
    return plant(x, planted, dtype)


def chain_tokens(rng, parent, parent_argmax_of, p_match, V):
    """Token of each non-root node: the parent's planted argmax with
    probability ``p_match[i]``, otherwise a uniform random token."""
    n = parent.size
    tok = np.empty(n, np.int32)
    u = rng.random(n)
    rnd = rng.integers(0, V, n, dtype=np.int32)
    for i in range(n):
        if parent[i] < 0:
            tok[i] = rnd[i]
        else:
            tok[i] = parent_argmax_of[parent[i]] if u[i] < p_match[i] else rnd[i]
    return tok


def attention_tensors(rng, n_nodes, prefix_tokens, Hq, Hkv, d, dtype):
    """q [n, Hq, d], k/v tree rows [n, Hkv, d], k/v prefix [P, Hkv, d], N(0,1)."""
    def draw(shape):
        if dtype == "bf16":
            return normal_bf16(rng, shape)
        return rng.standard_normal(size=shape, dtype=np.float32)
    return dict(q=draw((n_nodes, Hq, d)), k_tree=draw((n_nodes, Hkv, d)),
                v_tree=draw((n_nodes, Hkv, d)), k_pre=draw((prefix_tokens, Hkv, d)),
                v_pre=draw((prefix_tokens, Hkv, d)))


# ---------------------------------------------------------------------------
# workload 1: tiny tree verify
# ---------------------------------------------------------------------------
def tiny_tree(step: int = 0, V: int = 1000, P: int = 128, N: int = 60, Hq: int = 4,
              Hkv: int = 1, d: int = 64, k: int = 8, max_depth: int = 8,
              p_match: float = 0.7) -> dict:
    rng = make_rng(1, step)
    parent = random_tree(rng, N, max_depth)
    planted = rng.integers(0, V, N, dtype=np.int32)
    tok = chain_tokens(rng, parent, planted, np.full(N, p_match), V)
    logits = logits_rows(rng, N, V, 1.0, planted, "f32")
    att = attention_tensors(rng, N, P, Hq, Hkv, d, "f32")
    adj = rng.integers(0, V, (V, k), dtype=np.int32)
    return dict(workload="tiny_tree", dtype="f32", V=V, k=k, B=1, Hq=Hq, Hkv=Hkv, d=d,
                parent=parent, tok=tok, planted=planted, logits=logits, adj=adj,
                node_off=np.array([0, N], np.int32), pre_off=np.array([0, P], np.int32),
                vis_prefix=None, **att)


# ---------------------------------------------------------------------------
# workload 2: Graft-shaped single request (stateful, several steps)
# ---------------------------------------------------------------------------
def graft_static(V: int = QWEN3_VOCAB, k: int = 8) -> dict:
    """State shared by every step: the successor map g used to plant the
    target's argmax and the initial (uniform random) successor table."""
    rng = make_rng(2, 999_999)
    g = rng.integers(0, V, V, dtype=np.int32)
    adj0 = rng.integers(0, V, (V, k), dtype=np.int32)
    return dict(g=g, adj0=adj0, V=V, k=k)


def graft_step(step: int, static: dict, P: int = 2048, Hq: int = 32, Hkv: int = 8,
               d: int = 128, max_depth: int = 8, p_match: float = 0.7,
               p_follow: float = 0.8, budget: int = GRAFT_BUDGET) -> dict:
    """Draft part of one Graft verification step plus every random draw the
    step needs.  The retrieval tokens are not known here: they come from the
    successor table, after which ``graft_logits`` plants the target argmax."""
    V, g = static["V"], static["g"]
    rng = make_rng(2, step)
    stage = int(rng.integers(0, 4))
    nd = GRAFT_STAGE_DRAFT[stage]
    N = 1 + budget
    # draft nodes hang under the root: node 0 = root, nodes 1..nd drafts
    parent_d = random_tree(rng, 1 + nd, max_depth)
    root_tok = np.int32(rng.integers(0, V))
    follow_u = rng.random(N)
    follow_rnd = rng.integers(0, V, N, dtype=np.int32)
    # draft tokens: child = parent's planted argmax with p_match
    tok_d = np.empty(1 + nd, np.int32)
    tok_d[0] = root_tok
    planted_d = np.empty(1 + nd, np.int32)
    u = rng.random(1 + nd)
    rnd = rng.integers(0, V, 1 + nd, dtype=np.int32)
    for i in range(1 + nd):
        if i > 0:
            pa = planted_d[parent_d[i]]
            tok_d[i] = pa if u[i] < p_match else rnd[i]
        planted_d[i] = g[tok_d[i]] if follow_u[i] < p_follow else follow_rnd[i]
    noise = rng.standard_normal(size=(N, V), dtype=np.float32) * np.float32(2.0)
    att = attention_tensors(rng, N, P, Hq, Hkv, d, "bf16")
    return dict(workload="graft_hybrid", dtype="bf16", V=V, k=static["k"], B=1,
                Hq=Hq, Hkv=Hkv, d=d, stage=stage, n_draft=nd, N=N,
                parent_draft=parent_d, tok_draft=tok_d, root_tok=root_tok,
                follow_u=follow_u, follow_rnd=follow_rnd, noise=noise,
                node_off=np.array([0, N], np.int32), pre_off=np.array([0, P], np.int32),
                vis_prefix=None, **att)


def graft_logits(step_data: dict, static: dict, tok: np.ndarray) -> np.ndarray:
    """bf16 logits of all nodes once their tokens are known: node i's planted
    argmax is g[tok[i]] with probability 0.8, else a pre-drawn random token."""
    follow = step_data["follow_u"] < 0.8
    planted = np.where(follow, static["g"][tok], step_data["follow_rnd"]).astype(np.int32)
    return plant(step_data["noise"], planted, "bf16"), planted


# ---------------------------------------------------------------------------
# workload 3: D-cut batched block verify
# ---------------------------------------------------------------------------
def dcut_batch(step: int = 0, B: int = 64, D: int = 15, P_min: int = 512, P_max: int = 4096,
               V: int = QWEN3_VOCAB, Hq: int = 32, Hkv: int = 8, d: int = 128,
               with_attention: bool = True, with_logits: bool = True) -> dict:
    rng = make_rng(3, step)
    plen = rng.integers(P_min, P_max + 1, B).astype(np.int32)
    conf = rng.beta(4.0, 1.5, (B, D)).astype(np.float32)
    N = D + 1
    parent_1 = np.arange(-1, N - 1, dtype=np.int32)
    parent = np.tile(parent_1, B)
    planted = rng.integers(0, V, B * N, dtype=np.int32)
    u = rng.random((B, D))
    rnd = rng.integers(0, V, (B, N), dtype=np.int32)
    tok = rnd.copy()
    pl = planted.reshape(B, N)
    for j in range(1, N):
        tok[:, j] = np.where(u[:, j - 1] < conf[:, j - 1], pl[:, j - 1], rnd[:, j])
    out = dict(workload="dcut_batch", dtype="bf16", V=V, B=B, D=D, Hq=Hq, Hkv=Hkv, d=d,
               prefix_len=plen, conf=conf, rho=np.array(DCUT_RHOS, np.float32),
               parent=parent, tok=tok.reshape(-1).astype(np.int32), planted=planted,
               node_off=(np.arange(B + 1) * N).astype(np.int32),
               pre_off=np.concatenate([[0], np.cumsum(plen)]).astype(np.int32),
               vis_prefix=None)
    if with_logits:
        out["logits"] = logits_rows(rng, B * N, V, 2.0, planted, "bf16")
    if with_attention:
        out.update(attention_tensors(rng, B * N, int(plen.sum()), Hq, Hkv, d, "bf16"))
    return out


def successor_table(workload: int, V: int = QWEN3_VOCAB, k: int = 8) -> np.ndarray:
    """Initial V x k successor table with uniform random entries (the tables
    start untrained: no warm-up corpus is available)."""
    return make_rng(workload, 777_777).integers(0, V, (V, k), dtype=np.int32)


# ---------------------------------------------------------------------------
# workload 4: BlockPilot block-size sweep
# ---------------------------------------------------------------------------
def blockpilot_sweep(step: int = 0, B: int = 8, P: int = 8192, block: int = 16, half: int = 3,
                     V: int = QWEN3_VOCAB, hidden: int = 2048, Hq: int = 32, Hkv: int = 8,
                     d: int = 128, with_attention: bool = True, with_mlp: bool = True) -> dict:
    rng = make_rng(4, step)
    sizes = list(range(block - half, block + half + 1))
    n_out = len(sizes)
    # request tree: root, then one chain per block size, in increasing size
    parent_1 = [-1]
    leaf_1 = []
    for b in sizes:
        first = len(parent_1)
        parent_1.append(0)
        parent_1.extend(range(first, first + b - 1))
        leaf_1.append(len(parent_1) - 1)
    parent_1 = np.array(parent_1, np.int32)
    N = parent_1.size
    parent = np.tile(parent_1, B)
    planted = rng.integers(0, V, B * N, dtype=np.int32)
    conf = rng.beta(4.0, 1.5, B * N).astype(np.float32)
    tok = np.empty(B * N, np.int32)
    for r in range(B):
        sl = slice(r * N, (r + 1) * N)
        tok[sl] = chain_tokens(rng, parent_1, planted[sl], conf[sl], V)
    out = dict(workload="blockpilot_sweep", dtype="bf16", V=V, B=B, Hq=Hq, Hkv=Hkv, d=d,
               block=block, sizes=np.array(sizes, np.int32), hidden=hidden,
               parent=parent, tok=tok, planted=planted, conf=conf,
               leaf=np.array(leaf_1, np.int32), nodes_per_request=N,
               node_off=(np.arange(B + 1) * N).astype(np.int32),
               pre_off=(np.arange(B + 1) * P).astype(np.int32), vis_prefix=None)
    out["logits"] = logits_rows(rng, B * N, V, 2.0, planted, "bf16")
    out["last_logits"] = logits_rows(rng, B, V, 2.0, None, "bf16")
    if with_mlp:
        out["W1"] = normal_bf16(rng, (V, hidden), 0.02)
        out["W2"] = normal_bf16(rng, (hidden, n_out), 0.02)
        out["b1"] = np.zeros(hidden, np.float32)
        out["b2"] = np.zeros(n_out, np.float32)
    if with_attention:
        out.update(attention_tensors(rng, B * N, B * P, Hq, Hkv, d, "bf16"))
    return out


# ---------------------------------------------------------------------------
# workload 5: SpecOPD proposal-tree scoring
# ---------------------------------------------------------------------------
def specopd_tree(step: int = 0, prompt: int = 1024, response: int = 3072, n_anchor: int = 64,
                 W: int = 16, V: int = QWEN3_VOCAB, Hq: int = 32, Hkv: int = 8, d: int = 128,
                 with_attention: bool = True, with_logits: bool = True) -> dict:
    rng = make_rng(5, step)
    T = prompt + response
    anchors = np.sort(rng.choice(np.arange(prompt, T), n_anchor, replace=False)).astype(np.int32)
    N = n_anchor * W
    j = np.tile(np.arange(W, dtype=np.int32), n_anchor)
    node = np.arange(N, dtype=np.int32)
    parent = np.where(j == 0, -1, node - 1).astype(np.int32)
    vis_prefix = np.repeat(anchors + 1, W).astype(np.int32)
    branch_tok = rng.integers(0, V, N, dtype=np.int32)
    # the drafted next token that each node's distributions score
    mass_tok = np.where(j < W - 1, np.roll(branch_tok, -1), rng.integers(0, V, N)).astype(np.int32)
    out = dict(workload="specopd_tree", dtype="bf16", V=V, B=1, Hq=Hq, Hkv=Hkv, d=d,
               anchors=anchors, W=W, parent=parent, tok=branch_tok, mass_tok=mass_tok,
               vis_prefix=vis_prefix, node_off=np.array([0, N], np.int32),
               pre_off=np.array([0, T], np.int32),
               branch_off=(np.arange(n_anchor + 1) * W).astype(np.int32))
    if with_logits:
        out["lp"] = logits_rows(rng, N, V, 2.0, None, "bf16")
        out["lq"] = logits_rows(rng, N, V, 2.0, None, "bf16")
    if with_attention:
        out.update(attention_tensors(rng, N, T, Hq, Hkv, d, "bf16"))
    return out
