"""Workload 2 end to end: 200 seeded Graft verification steps, with the
successor table carried on the device from step to step, against the oracle
running the same 200 steps on its own copy of the table.

Graft page section 2, second and third gears: each step retrieves a subtree
from the V x 8 table, rooted at the current token and expanded by the
stage template; the hybrid tree (kept draft nodes + retrieved nodes, 61
nodes with the root) is verified in one pass; every verified position
rewrites the table row of its token with the target's top-8 next tokens, and
the next step retrieves from the updated table.  A stale or mis-ordered row
would show only here, where state crosses steps.

Per step and bit for bit: the retrieved tokens and parents, argmax / top-8 /
row max of all 61 logits rows, the accepted length, node, path and bonus
token, and the whole 151936 x 8 table; log-sum-exp within 1e-5; attention
(bf16, Qwen3-8B layer shape, prefix 2048) within 1e-2 * max|ref|.  The
oracle's attention runs in a process pool, one task per step.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import attn_close, dev, host, out_to_f64, sync
from oracle import accept as oacc
from oracle import graft as ogr
from oracle import vocab as ovoc
from oracle_pool import OraclePool, graft_attn_task

pytestmark = pytest.mark.gpu

STEPS = 200
K = 8
ATTN_BF16 = 1e-2
LSE_ATOL = 1e-5


def test_graft_workload_200_steps_table_carried(tv):
    st = synth.graft_static()
    V = st["V"]
    tp, tr, toff = tv.stage_templates()              # product's template data (host)
    otp, otr, ooff = ogr.stage_templates()           # the oracle's own derivation
    tmpl = [dev(x) for x in (tp, tr, toff)]
    adj_gpu = dev(st["adj0"])
    adj_ref = st["adj0"].copy()
    accepted = []
    with OraclePool() as pool:
        attn_ref = pool.imap(graft_attn_task, [(s, V) for s in range(STEPS)])
        for step in range(STEPS):
            d = synth.graft_step(step, st)
            stage, nd = d["stage"], d["n_draft"]
            S = ooff[stage + 1] - ooff[stage]
            N = d["N"]
            root = np.array([d["root_tok"]], np.int32)

            # ---- oracle chain on its own table
            ertok, erpar, ens = ogr.retrieve(adj_ref, root, np.array([stage]), otp, otr, ooff, 52)
            parent = ogr.assemble_hybrid(d["parent_draft"], otp[ooff[stage]:ooff[stage + 1]])
            tok = np.concatenate([d["tok_draft"], ertok[0, :S]]).astype(np.int32)
            logits, _ = synth.graft_logits(d, st, tok)
            ram, rti, rtv, rrm, rrl = ovoc.argmax_topk(logits, K)
            node_off = np.array([0, N], np.int32)
            ral, rbest, rpath, rbonus, _ = oacc.accept_longest_path(parent, tok, ram, node_off, None, 8)
            ogr.adj_update(adj_ref, tok, rti)

            # ---- CUDA chain on the device table
            rtok, rpar, ns, err = tv.graft_retrieve(adj_gpu, dev(root), dev(np.array([stage], np.int32)),
                                                    *tmpl, 52)
            tok_d = torch.cat([dev(d["tok_draft"]), rtok[0, :S]]).contiguous()
            par_d = dev(tv.assemble_hybrid(d["parent_draft"], tp[toff[stage]:toff[stage + 1]]))
            plen = dev(np.array([2048], np.int32))
            _, _, anc, _, _ = tv.tv_tree_prep(par_d, dev(node_off), plen, None, N, 1)
            o, lse = tv.tree_verify_attn(dev(d["q"]), dev(d["k_pre"]), dev(d["v_pre"]), dev(d["pre_off"]),
                                         dev(d["k_tree"]), dev(d["v_tree"]), dev(node_off), anc, N, 2048)
            am, ti, tvl, rm, rl = tv.vocab_argmax_topk(dev(logits), k=K)
            al, best, path, bonus, _ = tv.accept_longest_path(par_d, tok_d, am, dev(node_off), max_nodes=N,
                                                              max_depth=8)
            tv.graft_adj_update(adj_gpu, tok_d, ti)
            sync()

            where = f"step {step} (stage {stage}, {nd} draft nodes)"
            assert host(err)[0] == 0, where
            assert host(ns)[0] == ens[0] == S, where
            assert np.array_equal(host(rtok)[0, :S], ertok[0, :S]), where
            assert np.array_equal(host(rpar)[0, :S], erpar[0, :S]), where
            assert np.array_equal(host(tok_d), tok), where
            assert np.array_equal(host(am), ram), where
            assert np.array_equal(host(ti), rti), where
            assert np.array_equal(host(tvl), rtv), where
            assert np.array_equal(host(rm), rrm), where
            assert np.abs(host(rl).astype(np.float64) - rrl).max() <= LSE_ATOL, where
            assert host(al)[0] == ral[0] and host(best)[0] == rbest[0] and host(bonus)[0] == rbonus[0], where
            assert np.array_equal(host(path), rpath), where
            assert np.array_equal(host(adj_gpu), adj_ref), where

            s_ref, ro, rlse = next(attn_ref)
            assert s_ref == step
            ok, e, sc = attn_close(out_to_f64(o), ro, ATTN_BF16)
            assert ok, (where, e, sc)
            assert np.abs(host(lse) - rlse).max() <= 1e-4, where
            accepted.append(int(ral[0]))
    assert len(accepted) == STEPS and min(accepted) >= 0
