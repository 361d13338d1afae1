"""The allocation-free vocab reduction (vocab_argmax_topk_noalloc).

Callers such as runtimes with a fixed, pre-planned device-memory budget, or
serving loops whose allocator forbids cudaMalloc on the hot path, cannot hand
the library a workspace.  This entry point keeps its scratch in a fixed
device array inside the library.  Checked here through the C ABI against the
workspace-taking entry point and against the oracle, on two calls in a row
(the scratch keeps the previous call's contents), on both of its internal
paths (streamed chunks; the fallback for rows that are not 16-byte
multiples).  The file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import vocab as ovoc

pytestmark = pytest.mark.gpu

LSE_ATOL = 1e-5


@pytest.fixture(scope="module")
def tv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_tree_02_gb300 as m
    m.load_library()
    return m


def outputs(R, k, dev="cuda"):
    return (torch.full((R,), -1, dtype=torch.int32, device=dev),
            torch.full((R, k), -1, dtype=torch.int32, device=dev),
            torch.zeros((R, k), dtype=torch.float32, device=dev),
            torch.zeros(R, dtype=torch.float32, device=dev),
            torch.zeros(R, dtype=torch.float32, device=dev))


def against_oracle(host_logits, got, k, rows=None):
    sel = np.arange(host_logits.shape[0]) if rows is None else rows
    ram, rti, rtv, rrm, rrl = ovoc.argmax_topk(host_logits, k, rows=sel)
    am, ti, tvl, rm, rl = (t.cpu().numpy() for t in got)
    assert np.array_equal(am[sel], ram)
    assert np.array_equal(ti[sel], rti) and np.array_equal(tvl[sel], rtv)
    assert np.array_equal(rm[sel], rrm)
    assert np.abs(rl[sel].astype(np.float64) - rrl).max() <= LSE_ATOL


# (61, 151936, bf16): the Graft single-request rows; (300, 20000, bf16, k=16);
# (60, 1000, f32) and (7, 1001, f32): rows of 1001 floats are not 16-byte
# multiples, so that call takes the fallback kernels and their records
@pytest.mark.parametrize("rows,V,k,dtype", [(61, synth.QWEN3_VOCAB, 8, "bf16"), (300, 20000, 16, "bf16"),
                                            (60, 1000, 8, "f32"), (7, 1001, 8, "f32")])
def test_noalloc_matches_workspace_entry_point_and_oracle_twice(tv, rows, V, k, dtype):
    for call in range(2):
        rng = np.random.default_rng(100 * call + rows)
        x = (rng.standard_normal((rows, V)) * 2).astype(np.float32)
        host = synth.bf16_bits(x) if dtype == "bf16" else x
        L = torch.from_numpy(host.view(np.int16) if dtype == "bf16" else host).cuda()
        ref = tv.vocab_argmax_topk(L, k=k)
        got = tv.vocab_argmax_topk_noalloc(L, *outputs(rows, k), k=k)
        torch.cuda.synchronize()
        for a, b in zip(ref[:4], got[:4]):
            assert torch.equal(a, b)                       # integer results and max: bit-exact
        assert torch.allclose(ref[4], got[4], rtol=0, atol=LSE_ATOL)
        against_oracle(host, got, k)


def test_noalloc_row_gather(tv):
    d = synth.dcut_batch(B=5, V=12000, with_attention=False)
    L = torch.from_numpy(d["logits"].view(np.int16)).cuda()
    idx = np.array([3, 9, 40, 77, 79], np.int32)
    ref = tv.vocab_argmax_topk(L, k=8, row_idx=torch.from_numpy(idx).cuda(), out_rows=80)
    got = tv.vocab_argmax_topk_noalloc(L, *outputs(80, 8), k=8, row_idx=torch.from_numpy(idx).cuda())
    torch.cuda.synchronize()
    sel = torch.from_numpy(idx).long().cuda()
    for a, b in zip(ref[:4], got[:4]):
        assert torch.equal(a[sel], b[sel])
    against_oracle(d["logits"], got, 8, rows=idx)


def test_noalloc_rejects_sizes_beyond_its_scratch(tv):
    # the first row count whose scratch need exceeds the fixed array (k = 16,
    # the largest per-row need); the buffers are real and sized for the call
    # (about 4 GB of logits), and the entry point must refuse it on the host
    # (TV_EWORKSPACE) before any launch
    lib = tv.load_library()
    V, k = synth.QWEN3_VOCAB, 16
    lo, hi = 1, 65535
    while lo < hi:                                        # largest accepted row count
        mid = (lo + hi + 1) // 2
        if lib.vocab_argmax_topk_workspace_size(mid, V, k) <= (32 << 20):
            lo = mid
        else:
            hi = mid - 1
    rows = lo + 1
    assert lib.vocab_argmax_topk_workspace_size(rows, V, k) > (32 << 20)
    L = torch.zeros((rows, V), dtype=torch.bfloat16, device="cuda")
    am, ti, tvl, rm, rl = outputs(rows, k)
    with pytest.raises(tv.TVError) as e:
        tv.vocab_argmax_topk_noalloc(L, am, ti, tvl, rm, rl, k=k)
    assert e.value.status == -4
    torch.cuda.synchronize()
    assert bool((am == -1).all())                         # nothing was written
    del L
