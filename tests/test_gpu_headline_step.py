"""The D-cut batch-64 verification step exactly as bench.py times it: the
same entry points, launch configuration, buffers and CUDA graph
(``bench.make_step`` captured by ``bench.capture``), on the full-size
workload (64 requests of 1 + 15 nodes over 512..4096-token prefixes,
151936-entry bf16 logits, rho = 0.5), every output against the oracle.

D-cut page, technical summary: prefix-product scores, batch-global top-rho
selection, then verification of the kept positions only.  Graft page
section 2: every verified position updates its token's table row; the next
step retrieves from the bonus token.
"""
import numpy as np
import pytest
import torch

import bench
import synth
from gpu_util import attn_close, host, out_to_f64
from oracle import accept as oacc
from oracle import dcut as odc
from oracle import graft as ogr
from oracle import vocab as ovoc
from oracle_pool import oracle_attention_all

pytestmark = pytest.mark.gpu

RHO = 0.5


@pytest.fixture(scope="module")
def workload():
    d = synth.dcut_batch(step=0)
    adj0 = synth.successor_table(3)
    rhos = list(synth.DCUT_RHOS)
    ri = rhos.index(RHO)
    rs, rkeep, rkl, rpo, rpi = odc.select(d["conf"], rhos)
    K = int(rpo[ri, -1])
    rows = rpi[ri, :K]
    ram_k, rti_k, rtv_k, _, _ = ovoc.argmax_topk(d["logits"], 8, rows=rows)
    n = d["parent"].size
    ram = np.full(n, -1, np.int32)
    rti = np.zeros((n, 8), np.int32)
    ram[rows], rti[rows] = ram_k, rti_k
    ral, rbest, rpath, rbonus, rpacc = oacc.accept_longest_path(d["parent"], d["tok"], ram, d["node_off"],
                                                                rkeep[ri].reshape(-1), d["D"])
    adj = ogr.adj_update(adj0.copy(), d["tok"], rti, rkeep[ri].reshape(-1))
    otp, otr, ooff = ogr.stage_templates()
    rrt, rrp, rns = ogr.retrieve(adj, rbonus, np.full(d["B"], 2), otp, otr, ooff, 52)
    ro, _ = oracle_attention_all(d, node_cnt=rkl[ri])
    ref = dict(score=rs, keep=rkeep, keep_len=rkl, pack_off=rpo, pack_idx=rpi, K=K, rows=rows, argmax=ram_k,
               topk=rti_k, topk_val=rtv_k, accept_len=ral, best=rbest, path=rpath, bonus=rbonus, adj=adj,
               rtok=rrt, rpar=rrp, nslots=rns, attn=ro)
    return d, adj0, ref


def device_inputs(d, adj0):
    hd = {k: bench.to_dev(d[k], torch) for k in ("conf", "parent", "tok", "node_off", "pre_off", "prefix_len",
                                                  "q", "k_pre", "v_pre", "k_tree", "v_tree", "logits")}
    hd["adj"] = bench.to_dev(adj0, torch)
    hd.update(B=d["B"], D=d["D"], max_prefix=int(d["prefix_len"].max()))
    return hd


def check(out, hd, ref, K):
    ri = list(synth.DCUT_RHOS).index(RHO)
    sc, keep, kl, po, pi = (host(t) for t in out["sel"])
    assert np.array_equal(sc, ref["score"])
    assert np.array_equal(keep, ref["keep"]) and np.array_equal(kl, ref["keep_len"])
    assert np.array_equal(po, ref["pack_off"]) and np.array_equal(pi, ref["pack_idx"])
    rows = ref["rows"]
    am, ti, tvl = host(out["voc"][0]), host(out["voc"][1]), host(out["voc"][2])
    assert np.array_equal(am[rows], ref["argmax"])
    assert np.array_equal(ti[rows], ref["topk"]) and np.array_equal(tvl[rows], ref["topk_val"])
    al, best, path, bonus, _ = (host(t) for t in out["acc"])
    assert np.array_equal(al, ref["accept_len"]) and np.array_equal(best, ref["best"])
    assert np.array_equal(path, ref["path"]) and np.array_equal(bonus, ref["bonus"])
    assert np.array_equal(host(hd["adj"]), ref["adj"])
    rt, rp, ns, err = (host(t) for t in out["retr"])
    assert err[0] == 0 and np.array_equal(ns, ref["nslots"])
    assert np.array_equal(rt, ref["rtok"]) and np.array_equal(rp, ref["rpar"])
    assert host(out["n_bad"])[0] == 0
    ok, e, s = attn_close(out_to_f64(out["attn_out"]), ref["attn"], 1e-2)
    assert ok, (e, s)
    assert K == ref["K"] == int(kl[ri].sum())


def test_bench_step_graph_matches_oracle(tv, workload):
    d, adj0, ref = workload
    hd = device_inputs(d, adj0)
    stream = torch.cuda.Stream()
    step, kernels, out, K = bench.make_step(tv, torch, hd, RHO)
    # bench.capture runs the step once, then captures it; replaying applies
    # the same table update a second time, which leaves the table unchanged
    g = bench.capture(torch, step, stream)
    for t in (out["acc"][0], out["acc"][3], out["retr"][0], out["attn_out"]):
        t.fill_(-7)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    check(out, hd, ref, K)


def test_bench_end_to_end_step_with_host_logits(tv, workload):
    # the e2e leg: logits in pinned host memory, read in place over the host link
    d, adj0, ref = workload
    hd = device_inputs(d, adj0)
    pinned = bench.to_dev(d["logits"], torch, pin=True)
    step, kernels, out, K = bench.make_step(tv, torch, hd, RHO, logits=pinned)
    step()
    torch.cuda.synchronize()
    check(out, hd, ref, K)
