"""A pool of CPU processes that runs the oracle over full-size workloads.

The oracle is plain single-threaded NumPy.  Comparing every output of a
full-size workload (1024 attention nodes over a 4096-token trunk, 1024 rows
of 151936 logits) takes minutes in one process, so the GPU parity tests
split the nodes or rows over worker processes.  Each worker runs the oracle
unchanged on its slice; nothing here computes any part of the method.

The workload's arrays are placed in shared memory once by the test process;
workers attach to them by name, so a task carries only node or row indices.
The pool is started with ``spawn``: a process forked after CUDA has been
initialised can hang.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

_W: dict = {}


def _attach(specs):
    from multiprocessing import shared_memory
    _W.clear()
    for k, (name, shape, dtype) in specs.items():
        if name is None:
            _W[k] = (None, None)
            continue
        shm = shared_memory.SharedMemory(name=name)
        _W[k] = (shm, np.ndarray(shape, dtype=dtype, buffer=shm.buf))


_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def _init(specs):
    _attach(specs)


def _a(k):
    return _W[k][1] if k in _W else None


# ------------------------------------------------------------------ tasks
def attn_task(nodes):
    """Oracle attention output and lse of the given global nodes."""
    from oracle import attention as oatt
    o, lse = oatt.tree_attention(_a("q"), _a("k_pre"), _a("v_pre"), _a("pre_off"), _a("k_tree"), _a("v_tree"),
                                 _a("node_off"), _a("parent"), _a("vis_prefix"), node_cnt=_a("node_cnt"),
                                 nodes=nodes)
    return nodes, o[nodes], lse[nodes]


def vocab_task(args):
    """Oracle argmax / top-k / max / lse of the given rows of ``logits``."""
    from oracle import vocab as ovoc
    rows, k = args
    return rows, ovoc.argmax_topk(_a("logits"), k, rows=rows)


def alpha_task(rows):
    """Oracle alpha and softmax mass of the given rows of ``lp``/``lq``."""
    from oracle import alpha as oal
    mt = _a("mass_tok")
    a, _, _, pm = oal.tv_alpha(_a("lp"), _a("lq"), None, mt, rows=rows)
    return rows, a[rows], (None if pm is None else pm[rows])


def graft_attn_task(args):
    """Oracle attention of one Graft verification step (all 61 nodes).  The
    step's inputs are regenerated from its seed; the tree shape depends only
    on the step's pruning stage and draft tree, not on the successor table."""
    import synth
    from oracle import attention as oatt
    from oracle import graft as ogr
    step, V = args
    if ("static", V) not in _W:
        _W[("static", V)] = (None, synth.graft_static(V=V))
    d = synth.graft_step(step, _W[("static", V)][1])
    tp, _, off = ogr.stage_templates()
    st = d["stage"]
    parent = ogr.assemble_hybrid(d["parent_draft"], tp[off[st]:off[st + 1]])
    o, lse = oatt.tree_attention(d["q"], d["k_pre"], d["v_pre"], d["pre_off"], d["k_tree"], d["v_tree"],
                                 d["node_off"], parent)
    return step, o, lse


# ------------------------------------------------------------------ pool
class OraclePool:
    """``with OraclePool(arrays) as p: p.map(attn_task, chunks)``.

    ``arrays``: name -> ndarray or None (None reaches the task as None)."""

    def __init__(self, arrays: dict | None = None, workers: int | None = None):
        self.arrays = arrays or {}
        self.workers = workers or max(1, min(16, (os.cpu_count() or 2) - 1))
        self.shms = []
        self.pool = None

    def __enter__(self):
        from multiprocessing import shared_memory
        specs = {}
        for k, arr in self.arrays.items():
            if arr is None:
                specs[k] = (None, None, None)
                continue
            arr = np.ascontiguousarray(arr)
            shm = shared_memory.SharedMemory(create=True, size=max(1, arr.nbytes))
            np.ndarray(arr.shape, dtype=arr.dtype, buffer=shm.buf)[...] = arr
            self.shms.append(shm)
            specs[k] = (shm.name, arr.shape, arr.dtype.str)
        # one BLAS thread per worker: the variables must be in the environment
        # the workers start with (their NumPy is loaded before any initializer)
        saved = {k: os.environ.get(k) for k in _THREAD_VARS}
        os.environ.update({k: "1" for k in _THREAD_VARS})
        try:
            self.pool = mp.get_context("spawn").Pool(self.workers, initializer=_init, initargs=(specs,))
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        return self

    def map(self, fn, tasks):
        return self.pool.map(fn, tasks, chunksize=1)

    def imap(self, fn, tasks):
        return self.pool.imap(fn, tasks, chunksize=1)

    def __exit__(self, *exc):
        if self.pool is not None:
            self.pool.terminate() if exc[0] else self.pool.close()
            self.pool.join()
        for shm in self.shms:
            shm.close()
            shm.unlink()
        return False


def split(items, parts):
    """Contiguous slices of ``items`` (keeps nodes of one request together)."""
    items = list(items)
    n = max(1, min(parts, len(items)))
    bounds = np.linspace(0, len(items), n + 1).astype(int)
    return [items[bounds[i]:bounds[i + 1]] for i in range(n) if bounds[i + 1] > bounds[i]]


def oracle_attention_all(d, node_cnt=None, parts=96):
    """The oracle's attention for every node of workload ``d`` (only each
    request's first ``node_cnt[r]`` nodes when given; the others stay NaN),
    computed by a pool over contiguous node slices."""
    off = d["node_off"]
    n, Hq, dd = d["q"].shape
    nodes = list(range(n)) if node_cnt is None else [
        int(off[r]) + j for r in range(len(off) - 1) for j in range(int(node_cnt[r]))]
    keys = ("q", "k_pre", "v_pre", "pre_off", "k_tree", "v_tree", "node_off", "parent", "vis_prefix")
    arrays = {k: d.get(k) for k in keys}
    arrays["node_cnt"] = None if node_cnt is None else np.asarray(node_cnt, np.int32)
    ro = np.full((n, Hq, dd), np.nan)
    rlse = np.full((n, Hq), np.nan)
    with OraclePool(arrays) as pool:
        for idx, o, lse in pool.map(attn_task, split(nodes, parts)):
            ro[idx], rlse[idx] = o, lse
    return ro, rlse
