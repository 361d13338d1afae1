"""CPU oracle for batched speculative-tree verification — TEST INFRASTRUCTURE.

A plain, slow, obviously correct restatement of every step of the
verification path, in NumPy with fp64 arithmetic (except where a step's
result is defined in fp32: the D-cut prefix products).  It exists only to
check the CUDA library: the tests, ``__graft_entry__.smoke`` and the CPU
baseline leg of ``bench.py`` may import it; the product path never does, and
it shares no code with the CUDA library (the seeded input generators in
``synth`` are the only thing both consume).

Sources.  The method is described by four web pages; they are cited as
  * "Graft page"      — 浙江大学、阿里巴巴联手破解AI推理瓶颈 (write-up of
                        arXiv:2605.20104, Graft: pruning + retrieval grafting)
  * "BlockPilot page" — 阿里AMAP团队的AI提速新招："动态换挡"让大模型推理快4.2倍
                        (write-up of arXiv:2606.31315)
  * "D-cut page"      — D-cut: Adaptive Verification Depth Pruning for Batched
                        Speculative Decoding (gist.science summary)
  * "SpecOPD page"    — 【论文分享】给大模型推理安上"并发预读器": 解密阿里通义新作
                        SpecOPD ... (blog write-up of arXiv:2611.02846)
with the section of the page.

Modules
  tree       ancestor structure, depth and positions of a flattened tree
  attention  tree-masked grouped-query attention over a shared prefix
  vocab      per-row argmax / top-k / max / log-sum-exp
  alpha      alpha = 1 - TV(p, q), per-branch prefix product, softmax mass
  accept     greedy longest accepted path
  graft      successor-table update, stage templates, template retrieval
  dcut       prefix-product scores and batch-global budget selection
  mlp        BlockPilot block-size predictor

Parity status: every function is pinned by tests in ``tests/test_oracle_*.py``
except the *shape* of the Graft retrieval template, which the pages describe
only qualitatively (see ``graft.stage_template``: "parity unpinned" for the
template's exact slots; the retrieval given a template is pinned).
"""
from . import accept, alpha, attention, dcut, graft, mlp, tree, vocab  # noqa: F401

__all__ = ["accept", "alpha", "attention", "dcut", "graft", "mlp", "tree", "vocab"]
