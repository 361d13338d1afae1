"""Benchmark: batched speculative-tree verification on GB300 (libtreeverify).

Headline workload: D-cut batched block verify at batch 64 — each request a
chain of 1 bonus + 15 draft tokens over a prefix of 512..4096 tokens,
Qwen3-8B attention geometry (32 q heads, 8 KV heads, head_dim 128, bf16),
Qwen3 vocabulary (151936) bf16 logits.  One step = the whole verification
path for the batch:
  dcut_select -> tv_tree_prep -> tree_verify_attn (kept prefix of each chain)
  -> vocab_argmax_topk (kept rows, k = 8) -> accept_longest_path
  -> graft_adj_update (every verified node's top-8) -> graft_retrieve
     (next step's retrieval candidates from each request's bonus token)
Attention runs on a second stream beside the vocabulary chain (it shares
only the selection with it).  Metric: verified tree nodes per second (kept
positions per step / step time).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--rho 0.5] [--impl ours|reference]

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the same workload (a bounded sample of requests per step).
"""
from __future__ import annotations

import argparse
import json
import math
import re
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "verified tree nodes/s per GB300 at bs=64; HBM GB/s & TC util vs chip peak"
UNIT = "nodes/s"
L2_BYTES = 129 * 1024 * 1024
WORKLOAD = "dcut_batch_bs64"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--rho", type=float, default=0.5, help="D-cut budget ratio verified per step")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-rows", action="store_true", help="skip the per-row kernel measurements")
    ap.add_argument("--rows-only", default=None, help="regular expression: measure only the rows of these entry points")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d.get("bf16_tflops_sustained"),
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def config_dict(rho, n_gpus):
    return {"workload": WORKLOAD, "batch": 64, "draft_len": 15, "nodes_per_request": 16,
            "prefix_len": "uniform 512..4096", "attention": "32q/8kv heads, d=128, bf16",
            "vocab": synth.QWEN3_VOCAB, "topk": 8, "rho": rho, "rhos_selected": list(synth.DCUT_RHOS),
            "graft_table": "151936x8 int32", "retrieval_stage": "depth5 (20 slots)",
            "l2": "inputs exceed L2 (>700 MB read per step vs 129 MB L2); no flush needed",
            "parallelism": f"replicas x{n_gpus}" if n_gpus > 1 else "single GPU"}


# ============================================================ CPU oracle arm
# The oracle runs in spawned worker processes (single-threaded NumPy each).
# The workload's large arrays sit in shared memory, created once by the
# parent, so a task carries only indices: one kept position of one request
# (its attention over all heads and its vocabulary row).
_SHARED_KEYS = ("q", "k_pre", "v_pre", "k_tree", "v_tree", "logits", "pre_off", "parent")
_W = {}


def _worker_init(specs):
    from multiprocessing import shared_memory
    for k, (name, shape, dtype) in specs.items():
        shm = shared_memory.SharedMemory(name=name)
        _W[k] = (shm, np.ndarray(shape, dtype=dtype, buffer=shm.buf))


def _oracle_node(args):
    """Oracle of one kept position: tree attention of node (r, j) over its
    request's prefix and ancestors, all heads; argmax and top-8 of its logits."""
    r, j, N = args
    from oracle import attention as oatt, vocab as ovoc
    a = {k: v[1] for k, v in _W.items()}
    p0, p1 = int(a["pre_off"][r]), int(a["pre_off"][r + 1])
    sl = slice(r * N, (r + 1) * N)
    oatt.tree_attention(a["q"][sl], a["k_pre"][p0:p1], a["v_pre"][p0:p1], np.array([0, p1 - p0], np.int32),
                        a["k_tree"][sl], a["v_tree"][sl], np.array([0, N], np.int32), a["parent"][sl], nodes=[j])
    am, ti, _, _, _ = ovoc.argmax_topk(a["logits"][r * N + j:r * N + j + 1], 8)
    return int(am[0]), ti[0]


def oracle_step(d, reqs, pool, rho, adj, tmpl):
    """One oracle step on the kept positions of requests ``reqs`` (selection
    over the whole batch, then per position attention and vocabulary in the
    workers, then acceptance, table update and retrieval per request).
    Returns verified nodes."""
    from oracle import accept as oacc, dcut as odc, graft as ogr
    N = d["D"] + 1
    _, keep, keep_len, _, _ = odc.select(d["conf"], [rho])
    tasks = [(r, j, N) for r in reqs for j in range(int(keep_len[0, r]))]
    res = iter(pool.map(_oracle_node, tasks))
    nodes = 0
    tp, tr, off = tmpl
    for r in reqs:
        cnt = int(keep_len[0, r])
        argmax = np.full(N, -1, np.int32)
        ti = np.zeros((cnt, 8), np.int32)
        for j in range(cnt):
            argmax[j], ti[j] = next(res)
        sl = slice(r * N, (r + 1) * N)
        oacc.accept_longest_path(d["parent"][sl], d["tok"][sl], argmax, np.array([0, N], np.int32), keep[0, r])
        ogr.adj_update(adj, d["tok"][r * N:r * N + cnt], ti)
        ogr.retrieve(adj, d["tok"][[r * N]], np.full(1, 2), tp, tr, off, 52)
        nodes += cnt
    return nodes


def run_cpu_oracle(d, rho, steps, warmup, cores=None):
    """Time the oracle: W + K steps, each on the kept positions of cores / 8
    requests (7 i mod B for the i-th request taken).  Returns (nodes/s,
    cores, sample text, sec/step)."""
    from multiprocessing import shared_memory
    from oracle import graft as ogr
    tmpl = ogr.stage_templates()
    adj = synth.successor_table(3)
    if cores is None:
        cores = max(1, min(os.cpu_count() or 1, 16))
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    shms, specs = [], {}
    for k in _SHARED_KEYS:
        arr = np.ascontiguousarray(d[k])
        shm = shared_memory.SharedMemory(create=True, size=max(1, arr.nbytes))
        np.ndarray(arr.shape, dtype=arr.dtype, buffer=shm.buf)[...] = arr
        shms.append(shm)
        specs[k] = (shm.name, arr.shape, arr.dtype.str)
    ctx = mp.get_context("spawn")
    pool = ctx.Pool(cores, initializer=_worker_init, initargs=(specs,))
    B = d["B"]
    per = max(1, cores // 8)   # requests per step: about one kept position per worker
    reqs = lambda i: [(7 * (per * i + q)) % B for q in range(per)]
    try:
        oracle_step(d, [0], pool, rho, adj, tmpl)      # pool start-up
        for i in range(warmup):
            oracle_step(d, reqs(i), pool, rho, adj, tmpl)
        nodes, t = 0, 0.0
        for i in range(steps):
            a = time.perf_counter()
            nodes += oracle_step(d, reqs(warmup + i), pool, rho, adj, tmpl)
            t += time.perf_counter() - a
    finally:
        pool.close()
        pool.join()
        for shm in shms:
            shm.close()
            shm.unlink()
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    sample = (f"the kept positions of {per} request(s) per step (requests 7i mod 64; selection over the whole "
              f"batch), fp64 NumPy oracle, {cores} single-threaded worker processes, one position per task")
    return nodes / t, cores, sample, t / steps


# ============================================================ GPU arm
def to_dev(a, torch, pin=False):
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
    if pin:
        return t.pin_memory()
    return t.cuda()


def make_step(tv, torch, hd, rho, logits=None):
    """hd: dict of device tensors.  All outputs and workspaces are allocated
    here, once, so the step itself launches only libtreeverify kernels.
    ``logits``: the logits to verify against when not hd["logits"] (a pinned
    host tensor for the end-to-end step).  Returns (step_fn, kernels, out, K)."""
    logits = hd["logits"] if logits is None else logits
    B, D = hd["B"], hd["D"]
    N = D + 1
    V = synth.QWEN3_VOCAB
    rhos = list(synth.DCUT_RHOS)
    if rho not in rhos:
        rhos.append(rho)
    ri = rhos.index(rho)
    total = B * N
    K = int(math.floor(float(np.float32(rho)) * total + 0.5))
    tp, tr, toff = tv.stage_templates()
    tmpl = [to_dev(x, torch) for x in (tp, tr, toff)]
    stage = torch.full((B,), 2, dtype=torch.int32, device="cuda")
    max_prefix = int(hd["max_prefix"])
    lib = tv.load_library()
    e32 = lambda *s: torch.empty(s, dtype=torch.int32, device="cuda")
    out = {
        "sel": (torch.empty((B, N), dtype=torch.float32, device="cuda"),
                torch.empty((len(rhos), B, N), dtype=torch.uint8, device="cuda"),
                e32(len(rhos), B), e32(len(rhos), B + 1), e32(len(rhos), total)),
        "prep": (e32(total), e32(total), torch.empty((total, 1), dtype=torch.int64, device="cuda"),
                 e32(total), torch.zeros(1, dtype=torch.int32, device="cuda")),
        "attn_out": torch.empty_like(hd["q"]),
        "voc": (torch.full((total,), -1, dtype=torch.int32, device="cuda"), e32(total, 8),
                torch.empty((total, 8), dtype=torch.float32, device="cuda"), None, None),
        "acc": (e32(B), e32(B), e32(B, N), e32(B), e32(total)),
        "n_bad": torch.zeros(1, dtype=torch.int32, device="cuda"),
        "retr": (e32(B, 52), e32(B, 52), e32(B), torch.zeros(1, dtype=torch.int32, device="cuda")),
    }
    ws_attn = torch.empty(max(256, lib.tree_verify_attn_workspace_size(B, N, max_prefix, 32, 8, 128, 1)),
                          dtype=torch.uint8, device="cuda")
    ws_voc = torch.empty(max(256, lib.vocab_argmax_topk_workspace_size(K, V, 8)), dtype=torch.uint8,
                         device="cuda")
    sel = out["sel"]

    def k_dcut():
        tv.dcut_select(hd["conf"], rhos, outputs=sel)

    def k_prep():
        tv.tv_tree_prep(hd["parent"], hd["node_off"], hd["prefix_len"], None, N, 1, outputs=out["prep"])

    def k_attn():
        tv.tree_verify_attn(hd["q"], hd["k_pre"], hd["v_pre"], hd["pre_off"], hd["k_tree"], hd["v_tree"],
                            hd["node_off"], out["prep"][2], N, max_prefix, node_cnt=sel[2][ri],
                            out=out["attn_out"], want_lse=False, ws=ws_attn)

    def k_vocab():
        tv.vocab_argmax_topk(logits, k=8, rows=K, row_idx=sel[4][ri], out_rows=total,
                             want_lse=False, want_max=False, ws=ws_voc, outputs=out["voc"])

    def k_accept():
        tv.accept_longest_path(hd["parent"], hd["tok"], out["voc"][0], hd["node_off"], valid=sel[1][ri],
                               max_nodes=N, max_depth=D, outputs=out["acc"])

    def k_adj():
        tv.graft_adj_update(hd["adj"], hd["tok"], out["voc"][1], valid=sel[1][ri], n_bad=out["n_bad"])

    def k_retr():
        tv.graft_retrieve(hd["adj"], out["acc"][3], stage, *tmpl, 52, out=out["retr"])

    kernels = [("dcut_select", k_dcut, 1), ("tv_tree_prep", k_prep, 1),
               ("tree_verify_attn", k_attn, 1 + int(ws_attn.numel() > 256)),
               ("vocab_argmax_topk", k_vocab, 2), ("accept_longest_path", k_accept, 1),
               ("graft_adj_update", k_adj, 1), ("graft_retrieve", k_retr, 1)]

    # Dependencies: dcut_select and tv_tree_prep need nothing of each other;
    # tree_verify_attn needs both; the vocabulary pass needs only the kept
    # rows, and the acceptance / table update / retrieval chain needs only the
    # vocabulary results.  So attention runs on a second stream, forked after
    # the launch of dcut_select and joined at the end of the step, while the
    # vocabulary chain runs on the caller's stream.  The vocabulary pass is
    # captured before the attention launch so that its stream kernel takes
    # the SMs first and the attention CTAs fill them as it drains (the other
    # order measured 0.3-0.6 us slower).
    side = torch.cuda.Stream(priority=-1)
    ev_fork, ev_sel, ev_join = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()

    def step():
        cur = torch.cuda.current_stream()
        ev_fork.record(cur)
        side.wait_event(ev_fork)
        with torch.cuda.stream(side):
            k_prep()
        k_dcut()
        ev_sel.record(cur)
        k_vocab()
        with torch.cuda.stream(side):
            side.wait_event(ev_sel)
            k_attn()
            ev_join.record(side)
        k_accept()
        k_adj()
        k_retr()
        cur.wait_event(ev_join)
    return step, kernels, out, K


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = [l.split(", ") for l in (self.out or "").strip().splitlines() if l.strip()]
        rows = [r for r in rows if len(r) >= 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(rows[0][1]) if rows[0][1].replace(".", "").isdigit() else None,
                "reasons": reasons, "samples": len(rows)}


LAUNCH_REPS = 8    # calls per graph for the launch-bound rows
KERNEL_REPS = 4    # calls per graph for the per-kernel times of the step


def launch_us(torch, gr, stream):
    """Per-call time of a graph of LAUNCH_REPS calls."""
    return time_graph(torch, gr, 200, stream) / LAUNCH_REPS * 1e3


def time_graph(torch, graphs, n, stream):
    """Average duration of one replay; ``graphs`` (a graph or a list of graphs
    over distinct buffers) are replayed round-robin so that a working set
    smaller than L2 is not re-read from L2."""
    graphs = graphs if isinstance(graphs, list) else [graphs]
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):            # replay() launches on the current stream
        s.record(stream)
        for i in range(n):
            graphs[i % len(graphs)].replay()
        e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e) / n


def capture(torch, fn, stream, reps=1):
    """Graph of ``reps`` consecutive calls of ``fn``.  Replays of a graph
    complete on a cadence of about 2 us on this part, so a graph of one short
    kernel times the cadence, not the kernel; several calls per graph (they
    chain through programmatic launches, as inside the step) amortise it."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()                                   # first call outside the graph (lazy attributes)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(reps):
            fn()
    torch.cuda.synchronize()
    return g


def capture_seq(torch, fns, stream):
    """Graph of the calls ``fns`` in order (each called once outside the graph
    first), e.g. one call per buffer copy so that no call reads what the
    previous one left in L2."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for fn in fns:
            fn()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        for fn in fns:
            fn()
    torch.cuda.synchronize()
    return g


def copies_for(nbytes):
    """Distinct buffer copies needed for a rotation to exceed L2 twice over."""
    return max(1, min(32, math.ceil(2 * L2_BYTES / max(1, nbytes))))


def attn_bytes(plen, kept, Hq=32, Hkv=8, d=128):
    """Algorithmic bytes of one attention launch: every request's visible
    prefix K/V once, plus q, o and the own K/V row of each verified node."""
    kv = int(plen.sum()) * Hkv * d * 2 * 2
    return kv + int(kept) * (2 * Hq * d * 2 + 2 * Hkv * d * 2)


def sfu_ex2_per_s(torch):
    """Peak rate of 2^x on the special-function units: 16 results per clock
    per SM (4 per sub-partition) at the maximum SM clock."""
    p = torch.cuda.get_device_properties(torch.cuda.current_device())
    mhz = 2070.0
    mp = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(mp):
        mhz = float(json.load(open(mp)).get("sm_max_mhz", mhz))
    return 16.0 * p.multi_processor_count * mhz * 1e6


def row_entry(us, byts, pk, bound="hbm"):
    gbs = byts / us / 1e3
    return {"us": round(us, 2), "bytes": int(byts), "gbs": round(gbs, 1), "frac": round(gbs / pk["hbm"], 3),
            "bound": bound}


def measure_rows(tv, torch, pk, stream, only=None):
    """Rows of the path on their own workloads, timed with CUDA-graph replays
    (inputs rotated across enough copies to exceed L2).  `only`: a regular
    expression; rows whose entry-point names it does not match are skipped."""
    import re
    rows = {}

    def want(names):
        return only is None or any(re.search(only, n) for n in names.split("|"))

    g = torch.Generator(device="cuda")
    g.manual_seed(5005)
    V = synth.QWEN3_VOCAB
    bf = lambda *s, std=2.0: (torch.randn(s, generator=g, device="cuda") * std).to(torch.bfloat16)
    # a4: alpha on the SpecOPD scoring shape (1024 x 151936, two distributions)
    if want("tree_tv_alpha"):
        g.manual_seed(5005 + 0)   # each row draws its own inputs
        lp, lq = bf(1024, V), bf(1024, V)
        boff = torch.arange(0, 1025, 16, dtype=torch.int32, device="cuda")
        mtok = torch.randint(0, V, (1024,), generator=g, device="cuda", dtype=torch.int32)
        ws = torch.empty(tv.load_library().tree_tv_alpha_workspace_size(1024, V), dtype=torch.uint8, device="cuda")
        o3 = tuple(torch.empty(1024, dtype=torch.float32, device="cuda") for _ in range(3))
        gr = capture(torch, lambda: tv.tree_tv_alpha(lp, lq, boff, mtok, ws=ws, outputs=o3), stream,
                     reps=KERNEL_REPS)
        us = time_graph(torch, gr, 10, stream) * 1e3 / KERNEL_REPS
        e = row_entry(us, 2 * 1024 * V * 2, pk)
        # the special-function unit bounds this kernel: three exponentials per
        # vocabulary entry (the log-sum-exp of p and of q, then 2^min), 16 per
        # clock per SM
        n_ex2 = 3 * 1024 * V
        sfu_peak = sfu_ex2_per_s(torch)
        e.update(bound="sfu", ex2_per_s=round(n_ex2 / (us * 1e-6) / 1e12, 3), sfu_peak_ex2_per_s=round(sfu_peak / 1e12, 3),
                 frac_sfu=round(n_ex2 / (us * 1e-6) / sfu_peak, 3), frac_hbm=e["frac"])
        e["frac"] = e["frac_sfu"]
        rows["tree_tv_alpha[specopd 1024x151936 p,q bf16]"] = e
        del lp, lq, gr
    # a3: vocab reductions, Graft single request (61 rows) and D-cut batch (1024 rows)
    if want("vocab_argmax_topk"):
        g.manual_seed(5005 + 1)   # each row draws its own inputs
        for R in (61, 1024):
            nc = copies_for(R * V * 2)
            Ls = [bf(R, V) for _ in range(nc)]
            wsv = torch.empty(tv.load_library().vocab_argmax_topk_workspace_size(R, V, 8), dtype=torch.uint8,
                              device="cuda")
            outs = (torch.empty(R, dtype=torch.int32, device="cuda"), torch.empty((R, 8), dtype=torch.int32, device="cuda"),
                    torch.empty((R, 8), dtype=torch.float32, device="cuda"), torch.empty(R, dtype=torch.float32, device="cuda"),
                    torch.empty(R, dtype=torch.float32, device="cuda"))
            # graphs of several consecutive calls (as inside a step), each call
            # on its own copy of the logits so that none is served from L2
            reps = KERNEL_REPS if nc == 1 else min(KERNEL_REPS, nc)   # one copy: it exceeds L2 already
            grs = [capture_seq(torch, [lambda L=Ls[(i * reps + c) % nc]: tv.vocab_argmax_topk(L, k=8, ws=wsv, outputs=outs)
                                       for c in range(reps)], stream) for i in range(nc)]
            rows[f"vocab_argmax_topk[{R}x151936 bf16, k=8, max+lse]"] = row_entry(
                time_graph(torch, grs, 10 * nc, stream) * 1e3 / reps, R * V * 2, pk)
            del Ls, grs
    # a9: BlockPilot MLP (W1 151936 x 2048 bf16 = 622 MB)
    if want("blockpilot_mlp"):
        g.manual_seed(5005 + 2)   # each row draws its own inputs
        W1, W2, last = bf(V, 2048, std=0.02), bf(2048, 7, std=0.02), bf(8, V)
        lse = tv.vocab_argmax_topk(last, k=0)[4]
        wsm = torch.empty(tv.load_library().blockpilot_mlp_workspace_size(8, V, 2048), dtype=torch.uint8, device="cuda")
        om = (torch.empty((8, 7), dtype=torch.float32, device="cuda"), torch.empty(8, dtype=torch.int32, device="cuda"),
              torch.empty(8, dtype=torch.int32, device="cuda"))
        gr = capture(torch, lambda: tv.blockpilot_mlp(last, lse, W1, W2, ws=wsm, outputs=om), stream)
        rows["blockpilot_mlp[8x151936->2048->7]"] = row_entry(
            time_graph(torch, gr, 10, stream) * 1e3, V * 2048 * 2 + 8 * V * 2, pk)
        del W1, gr
    # a6 bulk form: whole-table update of 151936 rows from a [151936, 8] top-k array
    if want("graft_adj_update"):
        g.manual_seed(5005 + 3)   # each row draws its own inputs
        nbytes = V * 4 + 2 * V * 8 * 4
        nc = copies_for(nbytes)
        sets = [(torch.randint(0, V, (V, 8), generator=g, device="cuda", dtype=torch.int32),
                 torch.randperm(V, device="cuda", generator=g).to(torch.int32),
                 torch.randint(0, V, (V, 8), generator=g, device="cuda", dtype=torch.int32)) for _ in range(nc)]
        nb = torch.zeros(1, dtype=torch.int32, device="cuda")
        wsa = torch.empty(max(256, tv.load_library().graft_adj_update_workspace_size(V, V)), dtype=torch.uint8,
                          device="cuda")
        reps = min(KERNEL_REPS, nc)
        grs = [capture_seq(torch, [lambda a=a, t=t, k=k: tv.graft_adj_update(a, t, k, n_bad=nb, ws=wsa)
                                   for a, t, k in (sets[(i * reps + c) % nc] for c in range(reps))], stream)
               for i in range(nc)]
        rows["graft_adj_update[bulk 151936 rows x 8]"] = row_entry(
            time_graph(torch, grs, 10 * nc, stream) * 1e3 / reps, nbytes, pk)
        del sets, grs
    # a2 on the large-tree shapes, against the bf16 tensor peak: the SpecOPD
    # proposal tree (1024 nodes over one 4096-token trunk, 64 anchors) and the
    # BlockPilot sweep (8 requests x 8192-token prefix x 113 nodes)
    if want("tree_verify_attn"):
        g.manual_seed(5005 + 4)   # each row draws its own inputs
        for name, d in (("specopd 1024 nodes, trunk 4096", synth.specopd_tree(with_logits=False)),
                        ("blockpilot 8x(8192 prefix + 113 nodes)", synth.blockpilot_sweep(with_mlp=False, V=64))):
            rows[f"tree_verify_attn[{name}]"] = large_tree_row(tv, torch, d, pk, stream)
    # next rows, per-step planning kernels (kilobytes: launch-bound, reported in µs)
    if want("graft_stage_decide|graft_replace|dcut_choose_rho"):
        g.manual_seed(5005 + 5)   # each row draws its own inputs
        rng = np.random.default_rng(7007)
        B, S = 16, 60
        par = np.concatenate([synth.random_tree(rng, S, 8) for _ in range(B)]).astype(np.int32)
        conf = rng.beta(4.0, 1.5, B * S).astype(np.float32)
        tok = rng.integers(0, V, B * S).astype(np.int32)
        dp, dc, dt = to_dev(par, torch), to_dev(conf, torch), to_dev(tok, torch)
        doff = to_dev(np.arange(B + 1, dtype=np.int32) * S, torch)
        adj = to_dev(synth.successor_table(2), torch)
        tp, tr = tv.best_first_template(60)
        so = (torch.empty(B, dtype=torch.int32, device="cuda"), torch.empty((B, 3), dtype=torch.float32, device="cuda"),
              torch.zeros(1, dtype=torch.int32, device="cuda"))
        gr = capture(torch, lambda: tv.graft_stage_decide(dp, dc, doff, [0.6, 0.45, 0.2], max_nodes=S, outputs=so),
                     stream, reps=LAUNCH_REPS)
        rows["graft_stage_decide[16 trees x 60 nodes]"] = {"us": round(launch_us(torch, gr, stream), 2),
                                                           "bound": "launch"}
        ro = (torch.empty((B, S), dtype=torch.int32, device="cuda"), torch.empty((B, S), dtype=torch.int32, device="cuda"),
              torch.empty(B, dtype=torch.int32, device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda"))
        gr = capture(torch, lambda: tv.graft_replace(dp, dt, dc, S, 0.35, 0, adj, tp, tr, outputs=ro), stream,
                     reps=LAUNCH_REPS)
        rows["graft_replace[static, 16 trees x 60 slots]"] = {"us": round(launch_us(torch, gr, stream), 2),
                                                              "bound": "launch"}
        Bt, St = 64, 17
        tpar = to_dev(np.tile(np.arange(-1, St - 1, dtype=np.int32), Bt), torch)
        tconf = to_dev(rng.beta(4.0, 1.5, Bt * St).astype(np.float32), torch)
        ttok = to_dev(rng.integers(0, V, Bt * St).astype(np.int32), torch)
        to = (torch.empty((Bt, St), dtype=torch.int32, device="cuda"),
              torch.empty((Bt, St), dtype=torch.int32, device="cuda"),
              torch.empty(Bt, dtype=torch.int32, device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda"))
        gr = capture(torch, lambda: tv.graft_replace(tpar, ttok, tconf, St, 0.3, 1, adj, tp, tr, outputs=to), stream,
                     reps=LAUNCH_REPS)
        rows["graft_replace[TAIL, 64 blocks x 16 drafts]"] = {"us": round(launch_us(torch, gr, stream), 2),
                                                              "bound": "launch"}
        dconf = to_dev(synth.dcut_batch(with_attention=False, with_logits=False)["conf"], torch)
        sc, kp, *_ = tv.dcut_select(dconf, list(synth.DCUT_RHOS))
        gr = capture(torch, lambda: tv.dcut_choose_rho(sc, kp, [1.0, 1.35, 1.8, 2.4]), stream, reps=LAUNCH_REPS)
        rows["dcut_choose_rho[bs=64, 4 budgets]"] = {"us": round(launch_us(torch, gr, stream), 2),
                                                      "bound": "launch"}
    # T = 1 verification on the D-cut batch shape: 64 chains of 1 + 15 with
    # target and draft logits at every node (bf16, 151936); one CTA per
    # request walks its chain, each visited node costs vocabulary passes
    if want("accept_rejection_sampling"):
        g.manual_seed(5005 + 6)   # each row draws its own inputs
        Bs, Ns = 64, 16
        lg_p, lg_q = bf(Bs * Ns, V), bf(Bs * Ns, V)
        spar = to_dev(np.tile(np.arange(-1, Ns - 1, dtype=np.int32), Bs), torch)
        soff = to_dev(np.arange(Bs + 1, dtype=np.int32) * Ns, torch)
        stok = torch.randint(0, V, (Bs * Ns,), generator=g, device="cuda", dtype=torch.int32)
        su = torch.rand(Bs * Ns, generator=g, device="cuda") * 0.5        # about half the tests accept
        suf = torch.rand(Bs, generator=g, device="cuda")
        wss = torch.empty(tv.load_library().accept_rejection_sampling_workspace_size(Bs, V), dtype=torch.uint8,
                          device="cuda")
        souts = (torch.empty(Bs, dtype=torch.int32, device="cuda"), torch.empty(Bs, dtype=torch.int32, device="cuda"),
                 torch.empty((Bs, Ns), dtype=torch.int32, device="cuda"), torch.empty(Bs, dtype=torch.int32, device="cuda"))
        gr = capture(torch, lambda: tv.accept_rejection_sampling(spar, stok, lg_p, lg_q, soff, su, suf, max_nodes=Ns,
                                                                   max_depth=Ns - 1, ws=wss, outputs=souts), stream)
        us = time_graph(torch, gr, 20, stream) * 1e3
        acc_mean = float(souts[0].float().mean())
        rows["accept_rejection_sampling[T=1, 64 chains of 1+15, V=151936]"] = {
            "us": round(us, 2), "bound": "latency (sequential walk per request)", "mean_accept_len": round(acc_mean, 2)}
        del lg_p, lg_q
    return rows


def large_tree_row(tv, torch, d, pk, stream):
    """Attention on one large-tree workload: algorithmic flops = 4·d per
    (query head, node, visible key), visible keys = the node's visible prefix
    plus its ancestors (itself included)."""
    off, pre_off = d["node_off"], d["pre_off"]
    sizes, plen = np.diff(off), np.diff(pre_off).astype(np.int32)
    max_nodes, max_prefix = int(sizes.max()), int(plen.max())
    parent = d["parent"]
    depth = np.zeros(parent.size, np.int64)
    for i, p in enumerate(parent):          # parents precede children within a request
        if p >= 0:
            depth[i] = depth[off[np.searchsorted(off, i, side="right") - 1] + p] + 1
    vis = d["vis_prefix"] if d.get("vis_prefix") is not None else np.repeat(plen, sizes)
    n, Hq, dd = d["q"].shape
    Hkv = d["k_tree"].shape[1]
    flops = 4 * dd * Hq * int((vis.astype(np.int64) + depth + 1).sum())
    # bytes: each request's visible prefix K/V once per KV head, q, o, tree K/V
    kv_pre = sum(int(vis[off[r]:off[r + 1]].max()) for r in range(len(sizes))) * Hkv * dd * 2 * 2
    byts = kv_pre + n * (2 * Hq * dd * 2 + 2 * Hkv * dd * 2)
    one = sum(d[k].nbytes for k in ("q", "k_pre", "v_pre", "k_tree", "v_tree")) + d["q"].nbytes
    sets = []
    for _ in range(copies_for(one)):
        t = {k: to_dev(d[k], torch) for k in ("q", "k_pre", "v_pre", "k_tree", "v_tree")}
        t["out"] = torch.empty_like(t["q"])
        sets.append(t)
    dv = {k: to_dev(v, torch) for k, v in (("off", off), ("pre_off", pre_off), ("plen", plen),
                                            ("parent", parent), ("vis", vis.astype(np.int32)))}
    anc = tv.tv_tree_prep(dv["parent"], dv["off"], dv["plen"], dv["vis"], max_nodes, (max_nodes + 63) // 64)[2]
    ws = torch.empty(max(256, tv.load_library().tree_verify_attn_workspace_size(
        len(sizes), max_nodes, max_prefix, Hq, Hkv, dd, 1)), dtype=torch.uint8, device="cuda")
    grs = [capture(torch, lambda t=t: tv.tree_verify_attn(
        t["q"], t["k_pre"], t["v_pre"], dv["pre_off"], t["k_tree"], t["v_tree"], dv["off"], anc, max_nodes,
        max_prefix, vis_prefix=dv["vis"], out=t["out"], want_lse=False, ws=ws), stream) for t in sets]
    us = time_graph(torch, grs, 10 * len(sets), stream) * 1e3
    tfl = flops / us / 1e6
    return {"us": round(us, 2), "flops": flops, "tflops": round(tfl, 1), "frac": round(tfl / pk["bf16"], 3),
            "bound": "tensor", "bytes": byts, "gbs": round(byts / us / 1e3, 1)}


# ============================================================ per-config steps
def _step_row(torch, stream, sets, make, nodes, byts, pk, note):
    """Time one verification step of a workload.  ``sets``: input sets
    (rotated so that repeats are not served from L2); ``make(set)`` returns
    (step_fn, [(kernel name, fn, launches)]).  Reports the step time, verified
    nodes per second, the step's algorithmic bytes against HBM, and each
    kernel's time as a graph of KERNEL_REPS consecutive calls."""
    made = [make(t) for t in sets]
    grs = [capture(torch, m[0], stream) for m in made]
    us = time_graph(torch, grs, max(50, 10 * len(grs)), stream) * 1e3
    kern = {}
    for name, fn, _ in made[0][1]:
        gk = capture(torch, fn, stream, reps=KERNEL_REPS)
        kern[name] = round(time_graph(torch, gk, 50, stream) / KERNEL_REPS * 1e3, 2)
    return {"us": round(us, 2), "nodes": nodes, "nodes_per_s": round(nodes / us * 1e6, 1),
            "bytes": int(byts), "gbs": round(byts / us / 1e3, 1), "frac_hbm": round(byts / us / 1e3 / pk["hbm"], 3),
            "launches": sum(n for _, _, n in made[0][1]), "kernels_us": kern, "step": note}


def config_steps(tv, torch, pk, stream):
    """One verification step of each of the other four workloads, as CUDA
    graphs (the D-cut batch is the headline line itself)."""
    rows = {}
    i32 = lambda *s: torch.empty(s, dtype=torch.int32, device="cuda")
    V = synth.QWEN3_VOCAB
    lib = tv.load_library()

    def attn_call(t, n_nodes, max_nodes, max_prefix, B, Hq, Hkv, d, dt, vis=None, want_lse=False):
        ws = torch.empty(max(256, lib.tree_verify_attn_workspace_size(B, max_nodes, max_prefix, Hq, Hkv, d, dt)),
                         dtype=torch.uint8, device="cuda")
        out = torch.empty_like(t["q"])
        return lambda: tv.tree_verify_attn(t["q"], t["k_pre"], t["v_pre"], t["pre_off"], t["k_tree"], t["v_tree"],
                                           t["node_off"], t["anc"], max_nodes, max_prefix, vis_prefix=vis, out=out,
                                           want_lse=want_lse, ws=ws)

    def dev_set(d, keys):
        return {k: to_dev(d[k], torch) for k in keys}

    # ---- workload 1: tiny tree (V = 1000, prefix 128, 60 nodes, fp32, 4/1 heads, d = 64)
    d = synth.tiny_tree()
    n, P = d["parent"].size, int(d["pre_off"][1])
    keys = ("q", "k_pre", "v_pre", "k_tree", "v_tree", "logits", "parent", "tok", "adj", "node_off", "pre_off")
    one = sum(np.asarray(d[k]).nbytes for k in keys)

    def make1(t):
        t["plen"] = to_dev(np.array([P], np.int32), torch)
        prep_o = (i32(n), i32(n), torch.empty((n, 1), dtype=torch.int64, device="cuda"), i32(n),
                  torch.zeros(1, dtype=torch.int32, device="cuda"))
        t["anc"] = prep_o[2]
        attn = attn_call(t, n, n, P, 1, 4, 1, 64, 0)
        voc = (i32(n), i32(n, 8), torch.empty((n, 8), dtype=torch.float32, device="cuda"), None, None)
        wsv = torch.empty(lib.vocab_argmax_topk_workspace_size(n, 1000, 8), dtype=torch.uint8, device="cuda")
        acc = (i32(1), i32(1), i32(1, n), i32(1), None)
        nb = torch.zeros(1, dtype=torch.int32, device="cuda")
        ks = [("tv_tree_prep", lambda: tv.tv_tree_prep(t["parent"], t["node_off"], t["plen"], None, n, 1, outputs=prep_o), 1),
              ("tree_verify_attn", attn, 1),
              ("vocab_argmax_topk", lambda: tv.vocab_argmax_topk(t["logits"], k=8, want_lse=False, want_max=False,
                                                                  ws=wsv, outputs=voc), 3),
              ("accept_longest_path", lambda: tv.accept_longest_path(t["parent"], t["tok"], voc[0], t["node_off"],
                                                                     max_nodes=n, want_path_acc=False, outputs=acc), 1),
              ("graft_adj_update", lambda: tv.graft_adj_update(t["adj"], t["tok"], voc[1], n_bad=nb), 1)]

        def step():
            for _, f, _ in ks:
                f()
        return step, ks
    sets = [dev_set(d, keys) for _ in range(copies_for(one))]
    rows["step[tiny tree: 60 nodes, prefix 128, fp32 4/1 heads d=64, V=1000]"] = _step_row(
        torch, stream, sets, make1, n, one, pk, "tv_tree_prep -> tree_verify_attn (CUDA cores) -> vocab_argmax_topk "
        "-> accept_longest_path -> graft_adj_update")

    # ---- workload 2: Graft single request (61 nodes, prefix 2048, V = 151936, table carried)
    st = synth.graft_static()
    d = synth.graft_step(0, st)
    tp, tr, toff = tv.stage_templates()
    stage, nd, N = d["stage"], d["n_draft"], d["N"]
    tmpl = [to_dev(x, torch) for x in (tp, tr, toff)]
    parent = tv.assemble_hybrid(d["parent_draft"], tp[toff[stage]:toff[stage + 1]])
    adj = to_dev(st["adj0"], torch)
    # the target's logits for the tokens the first retrieval produces (fixed input)
    rt0 = tv.graft_retrieve(adj, to_dev(np.array([d["root_tok"]], np.int32), torch),
                            to_dev(np.array([stage], np.int32), torch), *tmpl, 52)[0]
    tok0 = np.concatenate([d["tok_draft"], rt0.cpu().numpy()[0, :N - 1 - nd]]).astype(np.int32)
    d["logits"], _ = synth.graft_logits(d, st, tok0)
    d["parent"] = parent
    keys = ("q", "k_pre", "v_pre", "k_tree", "v_tree", "logits", "parent", "node_off", "pre_off")
    one = sum(np.asarray(d[k]).nbytes for k in keys)
    root = to_dev(np.array([d["root_tok"]], np.int32), torch)
    stg = to_dev(np.array([stage], np.int32), torch)

    def make2(t):
        tokbuf = torch.zeros(1 + nd + 52, dtype=torch.int32, device="cuda")
        tokbuf[:1 + nd] = to_dev(d["tok_draft"], torch)
        tok = tokbuf[:N]
        rtok = tokbuf[1 + nd:].view(1, 52)
        retr = (rtok, i32(1, 52), i32(1), torch.zeros(1, dtype=torch.int32, device="cuda"))
        t["plen"] = to_dev(np.array([2048], np.int32), torch)
        prep_o = (i32(N), i32(N), torch.empty((N, 1), dtype=torch.int64, device="cuda"), i32(N),
                  torch.zeros(1, dtype=torch.int32, device="cuda"))
        t["anc"] = prep_o[2]
        attn = attn_call(t, N, N, 2048, 1, 32, 8, 128, 1)
        voc = (i32(N), i32(N, 8), torch.empty((N, 8), dtype=torch.float32, device="cuda"), None, None)
        wsv = torch.empty(lib.vocab_argmax_topk_workspace_size(N, V, 8), dtype=torch.uint8, device="cuda")
        acc = (i32(1), i32(1), i32(1, 9), i32(1), None)
        nb = torch.zeros(1, dtype=torch.int32, device="cuda")
        ks = [("graft_retrieve", lambda: tv.graft_retrieve(adj, root, stg, *tmpl, 52, out=retr), 1),
              ("tv_tree_prep", lambda: tv.tv_tree_prep(t["parent"], t["node_off"], t["plen"], None, N, 1,
                                                       outputs=prep_o), 1),
              ("tree_verify_attn", attn, 2),
              ("vocab_argmax_topk", lambda: tv.vocab_argmax_topk(t["logits"], k=8, want_lse=False, want_max=False,
                                                                  ws=wsv, outputs=voc), 3),
              ("accept_longest_path", lambda: tv.accept_longest_path(t["parent"], tok, voc[0], t["node_off"],
                                                                     max_nodes=N, max_depth=8, want_path_acc=False,
                                                                     outputs=acc), 1),
              ("graft_adj_update", lambda: tv.graft_adj_update(adj, tok, voc[1], n_bad=nb), 1)]

        def step():
            for _, f, _ in ks:
                f()
        return step, ks
    sets = [dev_set(d, keys) for _ in range(copies_for(one))]
    rows[f"step[graft: 61 nodes (stage {stage}), prefix 2048, 32/8 heads bf16, V=151936, table 151936x8]"] = _step_row(
        torch, stream, sets, make2, N, one + 52 * 4 + N * 8 * 4 * 2, pk,
        "graft_retrieve -> tv_tree_prep -> tree_verify_attn -> vocab_argmax_topk -> accept_longest_path -> "
        "graft_adj_update (the table carries from step to step)")
    del sets

    # ---- workload 4: BlockPilot sweep (8 x 113 nodes, prefix 8192, 7 block sizes)
    d = synth.blockpilot_sweep(with_mlp=False)
    n, Nr = d["parent"].size, d["nodes_per_request"]
    keys = ("q", "k_pre", "v_pre", "k_tree", "v_tree", "logits", "parent", "tok", "node_off", "pre_off")
    one = sum(np.asarray(d[k]).nbytes for k in keys)

    def make4(t):
        t["plen"] = to_dev(np.full(8, 8192, np.int32), torch)
        prep_o = (i32(n), i32(n), torch.empty((n, 2), dtype=torch.int64, device="cuda"), i32(n),
                  torch.zeros(1, dtype=torch.int32, device="cuda"))
        t["anc"] = prep_o[2]
        attn = attn_call(t, n, Nr, 8192, 8, 32, 8, 128, 1)
        voc = (i32(n), None, None, None, None)
        wsv = torch.empty(lib.vocab_argmax_topk_workspace_size(n, V, 0), dtype=torch.uint8, device="cuda")
        acc = (i32(8), i32(8), i32(8, 20), i32(8), i32(n))
        ks = [("tv_tree_prep", lambda: tv.tv_tree_prep(t["parent"], t["node_off"], t["plen"], None, Nr, 2,
                                                       outputs=prep_o), 1),
              ("tree_verify_attn", attn, 2),
              ("vocab_argmax_topk", lambda: tv.vocab_argmax_topk(t["logits"], k=0, want_lse=False, want_max=False,
                                                                  ws=wsv, outputs=voc), 3),
              ("accept_longest_path", lambda: tv.accept_longest_path(t["parent"], t["tok"], voc[0], t["node_off"],
                                                                     max_nodes=Nr, max_depth=19, outputs=acc), 1)]

        def step():
            for _, f, _ in ks:
                f()
        return step, ks
    sets = [dev_set(d, keys) for _ in range(copies_for(one))]
    rows["step[blockpilot: 8 x 113 nodes (7 block sizes), prefix 8192, 32/8 heads bf16, V=151936]"] = _step_row(
        torch, stream, sets, make4, n, one, pk,
        "tv_tree_prep -> tree_verify_attn -> vocab_argmax_topk (argmax) -> accept_longest_path (path_acc: the "
        "acceptance of all 7 block sizes); the block-size MLP runs once per request (its own row)")
    del sets

    # ---- workload 5: SpecOPD proposal tree (1024 nodes over a 4096-token trunk)
    d = synth.specopd_tree()
    n = d["parent"].size
    keys = ("q", "k_pre", "v_pre", "k_tree", "v_tree", "lp", "lq", "parent", "node_off", "pre_off", "vis_prefix",
            "branch_off", "mass_tok")
    one = sum(np.asarray(d[k]).nbytes for k in keys)

    def make5(t):
        t["plen"] = to_dev(np.array([4096], np.int32), torch)
        prep_o = (i32(n), i32(n), torch.empty((n, 16), dtype=torch.int64, device="cuda"), i32(n),
                  torch.zeros(1, dtype=torch.int32, device="cuda"))
        t["anc"] = prep_o[2]
        attn = attn_call(t, n, n, 4096, 1, 32, 8, 128, 1, vis=t["vis_prefix"])
        wsa = torch.empty(lib.tree_tv_alpha_workspace_size(n, V), dtype=torch.uint8, device="cuda")
        ao = tuple(torch.empty(n, dtype=torch.float32, device="cuda") for _ in range(3))
        ks = [("tv_tree_prep", lambda: tv.tv_tree_prep(t["parent"], t["node_off"], t["plen"], t["vis_prefix"], n, 16,
                                                       outputs=prep_o), 1),
              ("tree_verify_attn", attn, 2),
              ("tree_tv_alpha", lambda: tv.tree_tv_alpha(t["lp"], t["lq"], t["branch_off"], t["mass_tok"], ws=wsa,
                                                         outputs=ao), 1)]

        def step():
            for _, f, _ in ks:
                f()
        return step, ks
    sets = [dev_set(d, keys) for _ in range(copies_for(one))]
    rows["step[specopd: 1024 nodes (64 branches x 16), trunk 4096, 32/8 heads bf16, p,q V=151936]"] = _step_row(
        torch, stream, sets, make5, n, one, pk,
        "tv_tree_prep -> tree_verify_attn -> tree_tv_alpha (alpha, branch running product, softmax mass)")
    del sets
    return rows


# ============================================================ host memory placement
def _cpulist(text):
    out = set()
    for part in text.strip().split(","):
        if "-" in part:
            a, b = part.split("-")
            out.update(range(int(a), int(b) + 1))
        elif part:
            out.add(int(part))
    return out


def numa_report(torch, dev_index, buffers):
    """Where the end-to-end inputs live: the GPU's NUMA node (sysfs), the
    process's CPU affinity and the NUMA node of each CPU in it, and the nodes
    holding the pages of the given pinned buffers (/proc/self/numa_maps)."""
    rep = {}
    try:
        pr = torch.cuda.get_device_properties(dev_index)
        bus = f"{pr.pci_domain_id:04x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
        with open(f"/sys/bus/pci/devices/{bus}/numa_node") as f:
            rep["gpu_pci"], rep["gpu_numa_node"] = bus, int(f.read())
    except (OSError, AttributeError, ValueError, RuntimeError):
        rep["gpu_numa_node"] = None
    aff = sorted(os.sched_getaffinity(0))
    rep["cpu_affinity"] = f"{len(aff)} cpus ({aff[0]}-{aff[-1]})" if aff else "none"
    nodes = {}
    try:
        for nd in sorted(os.listdir("/sys/devices/system/node")):
            if nd.startswith("node") and nd[4:].isdigit():
                with open(f"/sys/devices/system/node/{nd}/cpulist") as f:
                    cpus = _cpulist(f.read())
                if cpus & set(aff):
                    nodes[int(nd[4:])] = len(cpus & set(aff))
    except OSError:
        pass
    rep["affinity_cpus_per_node"] = nodes
    # page placement of each buffer: numa_maps gives per-mapping page counts
    try:
        spans = []
        with open("/proc/self/maps") as f:
            for line in f:
                a, b = line.split()[0].split("-")
                spans.append((int(a, 16), int(b, 16)))
        counts = {}
        with open("/proc/self/numa_maps") as f:
            for line in f:
                parts = line.split()
                counts[int(parts[0], 16)] = {p.split("=")[0]: int(p.split("=")[1]) for p in parts[1:]
                                             if p.startswith("N") and "=" in p}
        pages = {}
        for t in buffers:
            addr = t.data_ptr()
            for a, b in spans:
                if a <= addr < b:
                    for k, v in counts.get(a, {}).items():
                        pages[k] = pages.get(k, 0) + v
                    break
        rep["pinned_pages_per_node"] = pages
    except OSError:
        rep["pinned_pages_per_node"] = None
    return rep


def max_over_ranks(x, dist, device):
    """The largest of every rank's x (the job's time is its slowest rank's)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, ms_step):
    """Units per second over all ranks: every replica verifies its own batch."""
    return world * units_per_rank / (ms_step / 1e3)


def gpu_arm(args):
    import torch
    import speculative_decoding_tree_02_gb300 as tv

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    pk = peaks()
    tv.load_library()

    d = synth.dcut_batch(step=0)
    plen = d["prefix_len"]
    hd = {k: to_dev(d[k], torch) for k in ("conf", "parent", "tok", "node_off", "pre_off", "prefix_len",
                                           "q", "k_pre", "v_pre", "k_tree", "v_tree", "logits")}
    hd["adj"] = to_dev(synth.successor_table(3), torch)
    hd.update(B=d["B"], D=d["D"], max_prefix=int(plen.max()))
    stream = torch.cuda.Stream()
    step, kernels, out, K = make_step(tv, torch, hd, args.rho)
    launches_per_step = sum(n for _, _, n in kernels)

    # graph of the whole step
    g_step = capture(torch, step, stream)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g_step.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk, torch.cuda.stream(stream):
        time.sleep(0.3)                         # let the sampler start before the timed region
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(args.steps):
            g_step.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), dist, "cuda")
    ms_step = ms_total / args.steps
    value = whole_job_rate(K, world, ms_step)

    # per-kernel graphs on the same buffers: average launch duration of each kernel
    per_kernel = {}
    for name, f, _ in kernels:
        gk = capture(torch, f, stream, reps=KERNEL_REPS)
        per_kernel[name] = time_graph(torch, gk, max(5, args.steps // 2), stream) / KERNEL_REPS
    a_bytes = attn_bytes(plen, K)           # |keep| = K exactly
    a_ms = per_kernel["tree_verify_attn"]
    traffic = load_traffic("tree_verify_attn", WORKLOAD)
    roofline = {"kernel": "tree_verify_attn", "bound": "hbm", "achieved": a_bytes / a_ms / 1e6,
                "peak": pk["hbm"], "unit": "GB/s", "frac": a_bytes / a_ms / 1e6 / pk["hbm"],
                "traffic": traffic, "algorithmic_bytes": a_bytes, "launch_us": a_ms * 1e3,
                "peak_source": f"{pk['src']} (MEASURED_PEAKS.json hbm_gbs, burst)"}
    v_bytes = K * synth.QWEN3_VOCAB * 2
    kern_json = {n: {"us": round(v * 1e3, 2)} for n, v in per_kernel.items()}
    kern_json["vocab_argmax_topk"].update(gbs=round(v_bytes / per_kernel["vocab_argmax_topk"] / 1e6, 1),
                                          frac=round(v_bytes / per_kernel["vocab_argmax_topk"] / 1e6 / pk["hbm"], 3))
    kern_json["tree_verify_attn"].update(gbs=round(roofline["achieved"], 1), frac=round(roofline["frac"], 3))

    # end to end through the C ABI with host buffers.  The step's inputs live
    # in pinned host memory.  Every step copies the small ones to the device;
    # the logits stay on the host and the vocabulary kernel reads the K kept
    # rows in place over the host link (the other rows never cross it).  The
    # results are read back to pinned host memory.
    step_inputs = ("conf", "parent", "tok", "q", "k_tree", "v_tree")
    pinned = {k: to_dev(d[k], torch, pin=True) for k in step_inputs + ("logits",)}
    h2d = sum(pinned[k].numel() * pinned[k].element_size() for k in step_inputs) + K * synth.QWEN3_VOCAB * 2
    # Two device input sets: step i's inputs are copied into set i & 1 on a
    # copy stream while step i - 1 runs; the steps themselves run in order on
    # one stream (the successor table is state carried from step to step).
    sets = [hd, dict(hd)]
    for k in step_inputs:
        sets[1][k] = torch.empty_like(hd[k])
    e2e_steps = [make_step(tv, torch, hs, args.rho, logits=pinned["logits"]) for hs in sets]
    graphs = [capture(torch, st[0], stream) for st in e2e_steps]
    copy_stream = torch.cuda.Stream()
    ev_copied = [torch.cuda.Event(), torch.cuda.Event()]
    ev_free = [torch.cuda.Event(), torch.cuda.Event()]   # the last step that used the set has finished
    for ev in ev_free:
        ev.record(stream)
    res_host = [{k: torch.empty(sz, dtype=torch.int32).pin_memory() for k, sz in
                 (("accept_len", (64,)), ("bonus", (64,)), ("path", (64, 16)), ("rtok", (64, 52)))} for _ in range(2)]
    d2h = sum(t.numel() * 4 for t in res_host[0].values())

    def e2e_step(i):
        b, out_b = i & 1, e2e_steps[i & 1][2]
        copy_stream.wait_event(ev_free[b])
        with torch.cuda.stream(copy_stream):
            for k in step_inputs:
                sets[b][k].copy_(pinned[k], non_blocking=True)
            ev_copied[b].record(copy_stream)
        stream.wait_event(ev_copied[b])
        with torch.cuda.stream(stream):
            graphs[b].replay()
            ev_free[b].record(stream)
            res_host[b]["accept_len"].copy_(out_b["acc"][0], non_blocking=True)
            res_host[b]["bonus"].copy_(out_b["acc"][3], non_blocking=True)
            res_host[b]["path"].copy_(out_b["acc"][2], non_blocking=True)
            res_host[b]["rtok"].copy_(out_b["retr"][0], non_blocking=True)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    n_e2e = max(3, min(args.steps, 20))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_host = time.perf_counter()
    e0.record(stream)
    copy_stream.wait_event(e0)
    for i in range(n_e2e):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    t_host = time.perf_counter() - t_host
    e2e_ms = max_over_ranks(max(e0.elapsed_time(e1), t_host * 1e3) / n_e2e, dist, "cuda")
    placement = numa_report(torch, local, list(pinned.values()))
    e2e = {"value": whole_job_rate(K, world, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
           "placement": placement,
           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
           "inputs": "pinned host memory; small inputs copied per step (overlapping the previous step), "
                     "logits read in place (only the kept rows cross the host link)"}

    rows = None
    if not args.no_rows and rank == 0:
        rows = measure_rows(tv, torch, pk, stream, only=args.rows_only)
        if args.rows_only is None or re.search(args.rows_only, "step"):
            rows.update(config_steps(tv, torch, pk, stream))

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded PCG64; shapes of the D-cut bs=64 workload)",
            "config": config_dict(args.rho, world), "roofline": roofline, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps, "kernels": kern_json,
            "clocks": clk.summary()}
    if rows:
        line["rows"] = rows
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample, _ = run_cpu_oracle(d, args.rho, steps=64, warmup=2)
        v1, _, sample1, _ = run_cpu_oracle(d, args.rho, steps=8, warmup=1, cores=1)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
                                "single_thread": {"value": v1, "unit": UNIT, "cores": 1, "sample": sample1}}
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


def load_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, when it was taken
    on the kernel as it is now (source hash match); else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        t = json.load(open(p)).get(f"{kernel}@{workload}")
    except (ValueError, OSError):
        return None
    if not t:
        return None
    return t["bytes_per_launch"] if source_hash(t["source"]) == t.get("source_sha") else None


def source_hash(sources):
    """First 16 hex digits of the SHA-256 over the named csrc files, in order
    (a comma-separated list), or None when one is missing."""
    import hashlib
    h = hashlib.sha256()
    for name in sources.split(","):
        p = os.path.join(ROOT, "speculative_decoding_tree_02_gb300", "csrc", name.strip())
        if not os.path.exists(p):
            return None
        h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def reference_arm(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    d = synth.dcut_batch(step=0)
    v, cores, sample, sec = run_cpu_oracle(d, args.rho, args.steps, args.warmup)
    line = {"metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded PCG64; shapes of the D-cut bs=64 workload)",
            "config": config_dict(args.rho, world), "impl": "reference",
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    args = parse()
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
