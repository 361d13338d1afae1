"""Python binding of libtreeverify (batched speculative-tree verification, sm_103a).

Each function here has the name of the C entry point it calls (see
``include/tv.h``) and only marshals arguments: it checks tensor devices and
dtypes, allocates outputs and workspaces with PyTorch (memory and streams are
PyTorch's job), passes raw pointers to the library on the current CUDA stream
and raises :class:`TVError` on a non-zero status.  Every step of the
computation runs in the library's CUDA kernels; there is no CPU fallback.
The library must have been built (``python -m speculative_decoding_tree_02_gb300.build``);
the first call raises if it is missing.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np
import torch

from .templates import stage_template, stage_templates, assemble_hybrid  # noqa: F401  (host-side template data)

__all__ = [
    "TVError", "lib", "tv_tree_prep", "tree_verify_attn", "vocab_argmax_topk", "vocab_argmax_topk_noalloc", "tree_tv_alpha",
    "accept_longest_path", "graft_adj_update", "graft_retrieve", "dcut_select", "blockpilot_mlp",
    "stage_templates", "assemble_hybrid", "LIB_PATH", "load_library", "EXPORTS",
    "graft_stage_decide", "graft_replace", "dcut_choose_rho", "best_first_template", "accept_rejection_sampling",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtreeverify.so")
TV_F32, TV_BF16 = 0, 1
MAX_NODES = 1024

_P, _I, _I64, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "tv_status_str": (ctypes.c_char_p, [_I]),
    "tv_version": (_I, []),
    "tv_tree_prep": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "tree_verify_attn_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "tree_verify_attn": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, ctypes.c_longlong,
                              ctypes.c_longlong, _I, _I, _I, _I, _F, _P, _P, _P, _SZ, _P]),
    "vocab_argmax_topk_workspace_size": (_SZ, [_I, _I, _I]),
    "vocab_argmax_topk": (_I, [_P, _I, _I, _I, _I64, _P, _I, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "vocab_argmax_topk_noalloc": (_I, [_P, _I, _I, _I, _I64, _P, _I, _P, _P, _P, _P, _P, _P]),
    "tree_tv_alpha_workspace_size": (_SZ, [_I, _I]),
    "tree_tv_alpha": (_I, [_P, _P, _I, _I, _I, _I64, _P, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "accept_longest_path": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "graft_adj_update_workspace_size": (_SZ, [_I, _I]),
    "graft_stage_decide": (_I, [_P, _P, _P, _I, _I, _P, _P, _P, _P, _P]),
    "graft_replace": (_I, [_P, _P, _P, _I, _I, ctypes.c_float, _I, _P, _I, _I, _P, _P, _I, _P, _P, _P, _P, _P]),
    "dcut_choose_rho": (_I, [_P, _P, _I, _I, _I, _P, _P, _P, _P]),
    "accept_rejection_sampling_workspace_size": (_SZ, [_I, _I]),
    "accept_rejection_sampling": (_I, [_P, _P, _P, _P, _I, _I, _I64, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P,
                                      _SZ, _P]),
    "graft_adj_update": (_I, [_P, _I, _I, _P, _P, _I, _P, _I, _P, _P, _SZ, _P]),
    "graft_retrieve": (_I, [_P, _I, _I, _P, _P, _I, _P, _P, _P, _I, _I, _P, _P, _P, _P, _P]),
    "dcut_select_workspace_size": (_SZ, [_I, _I, _I]),
    "dcut_select": (_I, [_P, _I, _I, _P, _I, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "blockpilot_mlp_workspace_size": (_SZ, [_I, _I, _I]),
    "blockpilot_mlp": (_I, [_P, _I64, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _SZ, _P]),
}
EXPORTS = tuple(_SIGS)
_LIB = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libtreeverify once; raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m speculative_decoding_tree_02_gb300.build` (needs nvcc)")
        handle = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = handle
    return _LIB


def __getattr__(name):
    if name == "lib":
        return load_library()
    raise AttributeError(name)


class TVError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {load_library().tv_status_str(status).decode()} ({status})")
        self.status = status


def _check(fn: str, status: int):
    if status != 0:
        raise TVError(fn, status)


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libtreeverify takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libtreeverify takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _ptr_dev_or_pinned(t: torch.Tensor):
    """Device tensor, or page-locked host tensor that the device reads in place."""
    if not t.is_cuda and not t.is_pinned():
        raise ValueError("expected a device tensor or a pinned host tensor")
    if not t.is_contiguous():
        raise ValueError("libtreeverify takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return TV_F32
    if t.dtype in (torch.bfloat16, torch.int16, torch.uint16):
        return TV_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: float32 or bfloat16")


def _i32(t: torch.Tensor, name: str):
    if t.dtype != torch.int32:
        raise TypeError(f"{name} must be int32")
    return t


def _ws(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# --------------------------------------------------------------------------- tree
def tv_tree_prep(parent, node_off, prefix_len, vis_prefix=None, max_nodes=None, anc_words=None,
                 outputs=None):
    """Returns depth, pos, anc (int64 view of the uint64 words), vis, err."""
    dev = parent.device
    B = node_off.numel() - 1
    n = parent.numel()
    if max_nodes is None:
        max_nodes = n
    W = anc_words or max(1, (max_nodes + 63) // 64)
    if outputs is None:
        depth = torch.empty(n, dtype=torch.int32, device=dev)
        pos = torch.empty_like(depth)
        vis = torch.empty_like(depth)
        anc = torch.empty((n, W), dtype=torch.int64, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    else:
        depth, pos, anc, vis, err = outputs
    _check("tv_tree_prep", load_library().tv_tree_prep(
        _ptr(_i32(parent, "parent")), _ptr(_i32(node_off, "node_off")), _ptr(_i32(prefix_len, "prefix_len")),
        _ptr(vis_prefix), B, max_nodes, W, _ptr(depth), _ptr(pos), _ptr(anc), _ptr(vis), _ptr(err), _stream()))
    return depth, pos, anc, vis, err


# ---------------------------------------------------------------------- attention
def tree_verify_attn(q, k_pre, v_pre, pre_off, k_tree, v_tree, node_off, anc, max_nodes, max_prefix,
                     vis_prefix=None, node_cnt=None, scale=None, out=None, lse=None, want_lse=True,
                     ws=None):
    n, Hq, d = q.shape
    Hkv = k_tree.shape[1]
    B = node_off.numel() - 1
    dt = _dtype_code(q)
    if scale is None:
        scale = 1.0 / d ** 0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((n, Hq), dtype=torch.float32, device=q.device)
    need = load_library().tree_verify_attn_workspace_size(B, max_nodes, max_prefix, Hq, Hkv, d, dt)
    if ws is None or ws.numel() < need:
        ws = _ws(need, q.device)
    _check("tree_verify_attn", load_library().tree_verify_attn(
        _ptr(q), _ptr(k_pre), _ptr(v_pre), _ptr(pre_off), _ptr(k_tree), _ptr(v_tree), _ptr(node_off),
        _ptr(node_cnt), _ptr(anc), anc.shape[1], _ptr(vis_prefix), B, max_nodes, max_prefix, n,
        k_pre.shape[0] if k_pre is not None else 0, Hq, Hkv, d, dt, float(scale), _ptr(out), _ptr(lse),
        _ptr(ws), ws.numel(), _stream()))
    return out, lse


# -------------------------------------------------------------------------- vocab
def vocab_argmax_topk(logits, k=8, rows=None, row_idx=None, out_rows=None, want_lse=True,
                      want_max=True, ws=None, outputs=None):
    """Outputs are indexed by source row; with ``row_idx`` give ``out_rows``
    (the output length, > max(row_idx)).  ``logits`` may be a pinned host
    tensor: the kernel then reads the rows it needs over the host link."""
    R, V = logits.shape
    dt = _dtype_code(logits)
    if rows is None:
        rows = row_idx.numel() if row_idx is not None else R
    n_out = out_rows if out_rows is not None else R
    dev = logits.device if logits.is_cuda else torch.device("cuda", torch.cuda.current_device())
    if outputs is None:
        argmax = torch.full((n_out,), -1, dtype=torch.int32, device=dev)
        tki = torch.empty((n_out, k), dtype=torch.int32, device=dev) if k else None
        tkv = torch.empty((n_out, k), dtype=torch.float32, device=dev) if k else None
        rmax = torch.empty(n_out, dtype=torch.float32, device=dev) if want_max else None
        rlse = torch.empty(n_out, dtype=torch.float32, device=dev) if want_lse else None
    else:
        argmax, tki, tkv, rmax, rlse = outputs
    need = load_library().vocab_argmax_topk_workspace_size(rows, V, k)
    if ws is None or ws.numel() < need:
        ws = _ws(need, dev)
    _check("vocab_argmax_topk", load_library().vocab_argmax_topk(
        _ptr_dev_or_pinned(logits), dt, rows, V, logits.stride(0), _ptr(row_idx), k, _ptr(argmax), _ptr(tki), _ptr(tkv),
        _ptr(rmax), _ptr(rlse), _ptr(ws), ws.numel(), _stream()))
    return argmax, tki, tkv, rmax, rlse


def vocab_argmax_topk_noalloc(logits, argmax, topk_idx=None, topk_val=None, row_max=None,
                              row_lse=None, k=8, rows=None, row_idx=None):
    """vocab_argmax_topk without a workspace (fixed device scratch inside the
    library, see include/tv.h); the caller passes preallocated outputs."""
    R, V = logits.shape
    if rows is None:
        rows = row_idx.numel() if row_idx is not None else R
    # outputs are indexed by source row: they must cover every row read
    need = rows
    if row_idx is not None and rows > 0 and not torch.cuda.is_current_stream_capturing():
        need = int(row_idx[:rows].max().item()) + 1
    for name, t, dt, cols in (("argmax", argmax, torch.int32, None), ("topk_idx", topk_idx, torch.int32, k),
                              ("topk_val", topk_val, torch.float32, k), ("row_max", row_max, torch.float32, None),
                              ("row_lse", row_lse, torch.float32, None)):
        if t is None:
            continue
        if t.dtype != dt or t.device != logits.device:
            raise ValueError(f"{name} must be a {dt} tensor on {logits.device}")
        if cols is not None and (t.dim() != 2 or t.shape[1] != cols):
            raise ValueError(f"{name} must have {cols} columns")
        if t.shape[0] < need:
            raise ValueError(f"{name} has {t.shape[0]} rows, the call writes row {need - 1}")
    _check("vocab_argmax_topk_noalloc", load_library().vocab_argmax_topk_noalloc(
        _ptr(logits), _dtype_code(logits), rows, V, logits.stride(0), _ptr(row_idx), k, _ptr(argmax),
        _ptr(topk_idx), _ptr(topk_val), _ptr(row_max), _ptr(row_lse), _stream()))
    return argmax, topk_idx, topk_val, row_max, row_lse


def tree_tv_alpha(lp, lq, branch_off=None, mass_tok=None, ws=None, outputs=None):
    R, V = lp.shape
    dt = _dtype_code(lp)
    dev = lp.device
    if outputs is None:
        alpha = torch.empty(R, dtype=torch.float32, device=dev)
        prefix = torch.empty_like(alpha) if branch_off is not None else None
        mass = torch.empty_like(alpha) if mass_tok is not None else None
    else:
        alpha, prefix, mass = outputs
    nb = branch_off.numel() - 1 if branch_off is not None else 0
    need = load_library().tree_tv_alpha_workspace_size(R, V)
    if ws is None or ws.numel() < need:
        ws = _ws(need, dev)
    _check("tree_tv_alpha", load_library().tree_tv_alpha(
        _ptr(lp), _ptr(lq), dt, R, V, lp.stride(0), _ptr(branch_off), nb, _ptr(mass_tok), _ptr(alpha),
        _ptr(prefix), _ptr(mass), _ptr(ws), ws.numel(), _stream()))
    return alpha, prefix, mass


# --------------------------------------------------------------------- acceptance
def accept_longest_path(parent, tok, argmax, node_off, valid=None, max_nodes=None, max_depth=None,
                        want_path_acc=True, outputs=None):
    dev = parent.device
    B = node_off.numel() - 1
    n = parent.numel()
    max_nodes = max_nodes or min(n, MAX_NODES)
    max_depth = max_nodes - 1 if max_depth is None else max_depth
    if outputs is None:
        accept_len = torch.empty(B, dtype=torch.int32, device=dev)
        best = torch.empty_like(accept_len)
        bonus = torch.empty_like(accept_len)
        path = torch.empty((B, max_depth + 1), dtype=torch.int32, device=dev)
        path_acc = torch.empty(n, dtype=torch.int32, device=dev) if want_path_acc else None
    else:
        accept_len, best, path, bonus, path_acc = outputs
    _check("accept_longest_path", load_library().accept_longest_path(
        _ptr(parent), _ptr(tok), _ptr(argmax), _ptr(valid), _ptr(node_off), B, max_nodes, max_depth,
        _ptr(accept_len), _ptr(best), _ptr(path), _ptr(bonus), _ptr(path_acc), _stream()))
    return accept_len, best, path, bonus, path_acc


# -------------------------------------------------------------------------- Graft
def graft_adj_update(adj, tok, topk_idx, valid=None, n_bad=None, ws=None):
    V, k = adj.shape
    n = tok.numel()
    if n_bad is None:
        n_bad = torch.zeros(1, dtype=torch.int32, device=adj.device)
    need = load_library().graft_adj_update_workspace_size(V, n)
    if need and (ws is None or ws.numel() < need):
        ws = torch.empty(need, dtype=torch.uint8, device=adj.device)
    _check("graft_adj_update", load_library().graft_adj_update(
        _ptr(adj), V, k, _ptr(tok), _ptr(topk_idx), topk_idx.stride(0), _ptr(valid), n, _ptr(n_bad),
        _ptr(ws) if need else None, ws.numel() if need else 0, _stream()))
    return n_bad


def graft_retrieve(adj, root_tok, stage, tparent, trank, tmpl_off, max_slots, out=None):
    V, k = adj.shape
    B = root_tok.numel()
    dev = adj.device
    if out is None:
        rtok = torch.empty((B, max_slots), dtype=torch.int32, device=dev)
        rpar = torch.empty_like(rtok)
        ns = torch.empty(B, dtype=torch.int32, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    else:
        rtok, rpar, ns, err = out
    _check("graft_retrieve", load_library().graft_retrieve(
        _ptr(adj), V, k, _ptr(root_tok), _ptr(stage), B, _ptr(tparent), _ptr(trank), _ptr(tmpl_off),
        tmpl_off.numel() - 1, max_slots, _ptr(rtok), _ptr(rpar), _ptr(ns), _ptr(err), _stream()))
    return rtok, rpar, ns, err


# -------------------------------------------------------------------------- D-cut
def dcut_select(conf, rhos: Sequence[float], outputs=None):
    B, D = conf.shape
    T = B * (D + 1)
    dev = conf.device
    n_rho = len(rhos)
    rho_host = (ctypes.c_float * n_rho)(*[float(r) for r in rhos])
    if outputs is None:
        score = torch.empty((B, D + 1), dtype=torch.float32, device=dev)
        keep = torch.empty((n_rho, B, D + 1), dtype=torch.uint8, device=dev)
        keep_len = torch.empty((n_rho, B), dtype=torch.int32, device=dev)
        pack_off = torch.empty((n_rho, B + 1), dtype=torch.int32, device=dev)
        pack_idx = torch.empty((n_rho, T), dtype=torch.int32, device=dev)
    else:
        score, keep, keep_len, pack_off, pack_idx = outputs
    _check("dcut_select", load_library().dcut_select(
        _ptr(conf), B, D, rho_host, n_rho, _ptr(score), _ptr(keep), _ptr(keep_len), _ptr(pack_off),
        _ptr(pack_idx), None, 0, _stream()))
    return score, keep, keep_len, pack_off, pack_idx


def dcut_choose_rho(score, keep, cost: Sequence[float]):
    """Expected tokens per budget (float64 [n_rho]) and rho* (int32 [1])."""
    n_rho, B, N = keep.shape
    cost_host = (ctypes.c_float * n_rho)(*[float(c) for c in cost])
    exp_tok = torch.empty(n_rho, dtype=torch.float64, device=score.device)
    rho_star = torch.empty(1, dtype=torch.int32, device=score.device)
    _check("dcut_choose_rho", load_library().dcut_choose_rho(
        _ptr(score), _ptr(keep), B, N - 1, n_rho, cost_host, _ptr(exp_tok), _ptr(rho_star), _stream()))
    return exp_tok, rho_star


def accept_rejection_sampling(parent, tok, p_logits, q_logits, node_off, u_node, u_final, max_nodes=None,
                              max_depth=None, ws=None, outputs=None):
    """T = 1 verification.  Returns accept_len, best_node int32 [B], path
    int32 [B, max_depth+1], bonus int32 [B]."""
    n, V = p_logits.shape
    B = node_off.numel() - 1
    dev = parent.device
    if max_nodes is None:
        max_nodes = n
    if max_depth is None:
        max_depth = max_nodes - 1
    dt = _dtype_code(p_logits)
    need = load_library().accept_rejection_sampling_workspace_size(B, V)
    if ws is None or ws.numel() < need:
        ws = _ws(need, dev)
    if outputs is None:
        acc = torch.empty(B, dtype=torch.int32, device=dev)
        best = torch.empty_like(acc)
        path = torch.empty((B, max_depth + 1), dtype=torch.int32, device=dev)
        bonus = torch.empty_like(acc)
    else:
        acc, best, path, bonus = outputs
    _check("accept_rejection_sampling", load_library().accept_rejection_sampling(
        _ptr(parent), _ptr(tok), _ptr(p_logits), _ptr(q_logits), dt, V, p_logits.stride(0), _ptr(node_off), B,
        max_nodes, max_depth, _ptr(u_node), _ptr(u_final), _ptr(acc), _ptr(best), _ptr(path), _ptr(bonus),
        _ptr(ws), ws.numel(), _stream()))
    return acc, best, path, bonus


# -------------------------------------------------------------- Graft planning
def best_first_template(S: int = 60, width: int = 8, depth: int = 8, device="cuda"):
    """(tparent, trank) int32 device tensors: the first S best-first rank paths."""
    tp, tr = stage_template(S, width, depth)
    return (torch.from_numpy(np.ascontiguousarray(tp)).to(device),
            torch.from_numpy(np.ascontiguousarray(tr)).to(device))


def graft_stage_decide(parent, conf, node_off, tau: Sequence[float], max_nodes=None, outputs=None):
    """Returns stage int32 [B], best float32 [B, 3], err int32 [1]."""
    B = node_off.numel() - 1
    if max_nodes is None:
        max_nodes = parent.numel()
    tau_host = (ctypes.c_float * 3)(*[float(x) for x in tau])
    if outputs is None:
        stage = torch.empty(B, dtype=torch.int32, device=parent.device)
        best = torch.empty((B, 3), dtype=torch.float32, device=parent.device)
        err = torch.zeros(1, dtype=torch.int32, device=parent.device)
    else:
        stage, best, err = outputs
    _check("graft_stage_decide", load_library().graft_stage_decide(
        _ptr(parent), _ptr(conf), _ptr(node_off), B, max_nodes, tau_host, _ptr(stage), _ptr(best), _ptr(err),
        _stream()))
    return stage, best, err


def graft_replace(parent, tok, conf, S: int, tau: float, attach: int, adj, tparent, trank, outputs=None):
    """Request r's tree = nodes r*S..r*S+S-1.  Returns tok_out, parent_out
    int32 [B, S], n_kept int32 [B], err int32 [1]."""
    B = tok.numel() // S
    V, k = adj.shape
    dev = tok.device
    if outputs is None:
        tok_out = torch.empty((B, S), dtype=torch.int32, device=dev)
        par_out = torch.empty((B, S), dtype=torch.int32, device=dev)
        n_kept = torch.empty(B, dtype=torch.int32, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    else:
        tok_out, par_out, n_kept, err = outputs
    _check("graft_replace", load_library().graft_replace(
        _ptr(parent), _ptr(tok), _ptr(conf), B, S, float(tau), int(attach), _ptr(adj), V, k, _ptr(tparent),
        _ptr(trank), tparent.numel(), _ptr(tok_out), _ptr(par_out), _ptr(n_kept), _ptr(err), _stream()))
    return tok_out, par_out, n_kept, err


# --------------------------------------------------------------------- BlockPilot
def blockpilot_mlp(last_logits, row_lse, W1, W2, b1=None, b2=None, block=16, ws=None, outputs=None):
    B, V = last_logits.shape
    H = W1.shape[1]
    C = W2.shape[1]
    dev = last_logits.device
    if outputs is None:
        z = torch.empty((B, C), dtype=torch.float32, device=dev)
        choice = torch.empty(B, dtype=torch.int32, device=dev)
        bsize = torch.empty_like(choice)
    else:
        z, choice, bsize = outputs
    need = load_library().blockpilot_mlp_workspace_size(B, V, H)
    if ws is None or ws.numel() < need:
        ws = _ws(need, dev)
    _check("blockpilot_mlp", load_library().blockpilot_mlp(
        _ptr(last_logits), last_logits.stride(0), _ptr(row_lse), _ptr(W1), _ptr(b1), _ptr(W2), _ptr(b2),
        B, V, H, C, block, _ptr(z), _ptr(choice), _ptr(bsize), _ptr(ws), ws.numel(), _stream()))
    return z, choice, bsize
