"""The allocation-free vocab reduction (vocab_argmax_topk_noalloc).

Callers such as runtimes with a fixed, pre-planned device-memory budget, or
serving loops whose allocator forbids cudaMalloc on the hot path, cannot hand
the library a workspace.  This entry point keeps its scratch in a fixed
device array inside the library.  Checked here through the C ABI against the
workspace-taking entry point, on two calls in a row (the scratch keeps the
previous call's contents).  The file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


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


@pytest.mark.parametrize("rows,V,k,dtype", [(61, synth.QWEN3_VOCAB, 8, "bf16"), (300, 20000, 16, "bf16"),
                                            (60, 1000, 8, "f32")])
def test_noalloc_matches_workspace_entry_point_twice(tv, rows, V, k, dtype):
    for call in range(2):
        rng = np.random.default_rng(100 * call + rows)
        x = (rng.standard_normal((rows, V)) * 2).astype(np.float32)
        host = synth.bf16_bits(x).view(np.int16) if dtype == "bf16" else x
        L = torch.from_numpy(host).cuda()
        ref = tv.vocab_argmax_topk(L, k=k)
        got = tv.vocab_argmax_topk_noalloc(L, *outputs(rows, k), k=k)
        torch.cuda.synchronize()
        for a, b in zip(ref[:4], got[:4]):
            assert torch.equal(a, b)                       # integer results and max: bit-exact
        assert torch.allclose(ref[4], got[4], rtol=0, atol=1e-5)


def test_noalloc_row_gather(tv):
    d = synth.dcut_batch(B=5, V=12000, with_attention=False)
    L = torch.from_numpy(d["logits"].view(np.int16)).cuda()
    idx = torch.tensor([3, 9, 40, 77, 79], dtype=torch.int32, device="cuda")
    ref = tv.vocab_argmax_topk(L, k=8, row_idx=idx, out_rows=80)
    got = tv.vocab_argmax_topk_noalloc(L, *outputs(80, 8), k=8, row_idx=idx)
    torch.cuda.synchronize()
    sel = idx.long()
    for a, b in zip(ref[:4], got[:4]):
        assert torch.equal(a[sel], b[sel])


def test_noalloc_rejects_sizes_beyond_its_scratch(tv):
    import ctypes
    lib = tv.load_library()
    need = lib.vocab_argmax_topk_workspace_size(20000, synth.QWEN3_VOCAB, 8)
    assert need > (32 << 20)
    status = lib.vocab_argmax_topk_noalloc(ctypes.c_void_p(256), 1, 20000, synth.QWEN3_VOCAB,
                                           synth.QWEN3_VOCAB, None, 8, ctypes.c_void_p(256),
                                           ctypes.c_void_p(256), None, None, None, None)
    assert status == -4                                   # TV_EWORKSPACE, nothing launched
