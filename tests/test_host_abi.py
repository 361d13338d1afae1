"""Host-side checks (no GPU): the C-ABI library builds, loads and exports every
entry point declared in include/tv.h, and the product's template builder
agrees with the oracle's independent derivation."""
import os
import re
import subprocess
import sys

import numpy as np
import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "tv.h")
LIB = os.path.join(ROOT, "speculative_decoding_tree_02_gb300", "libtreeverify.so")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def built_lib():
    if not os.path.exists(LIB):
        subprocess.run([sys.executable, "-m", "speculative_decoding_tree_02_gb300.build"], cwd=ROOT,
                       check=True)
    return LIB


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ["tv_tree_prep", "tree_verify_attn", "vocab_argmax_topk", "tree_tv_alpha",
                     "accept_longest_path", "graft_adj_update", "graft_retrieve", "dcut_select",
                     "blockpilot_mlp", "tv_status_str", "tv_version"]:
        assert required in names


def test_library_exports_every_declared_symbol(built_lib):
    out = subprocess.run(["nm", "-D", "--defined-only", built_lib], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing


def test_library_loads_and_binding_matches_header(built_lib):
    import speculative_decoding_tree_02_gb300 as tv
    lib = tv.load_library()
    assert lib.tv_version() >= 100
    assert lib.tv_status_str(-1).decode().startswith("TV_EINVAL")
    assert set(tv.EXPORTS) == set(declared_functions())


def validation_calls(lib, buf):
    """Calls that host validation must refuse (status, call) before any
    launch.  ``buf``: the pointer passed for every array argument."""
    import ctypes
    null = None
    rho = (ctypes.c_float * 1)(1.5)
    return [
        # k above the supported maximum
        (-2, lambda: lib.vocab_argmax_topk(buf, 1, 4, 100, 100, null, 17, buf, buf, null, null, null, buf,
                                           1 << 20, null)),
        # missing workspace
        (-4, lambda: lib.vocab_argmax_topk(buf, 1, 4, 100, 100, null, 8, buf, buf, null, null, null, null, 0,
                                           null)),
        # head dim not supported
        (-2, lambda: lib.tree_verify_attn(*([buf] * 9), 1, null, 1, 8, 8, 8, 8, 4, 1, 96, 1, ctypes.c_float(0.1),
                                          buf, null, null, 0, null)),
        # too many nodes per request
        (-2, lambda: lib.tv_tree_prep(*([buf] * 4), 1, 2000, 32, *([buf] * 5), null, null)),
        # rho outside [0, 1]
        (-1, lambda: lib.dcut_select(buf, 4, 3, rho, 1, *([buf] * 5), null, 0, null)),
        # zero-size calls are no-ops
        (0, lambda: lib.accept_longest_path(null, null, null, null, null, 0, 8, 8, null, null, null, null, null,
                                            null)),
    ]


def test_host_validation_rejects_bad_arguments_without_launching(built_lib):
    """Entry points validate on the host and return an error before any
    launch.  Without a GPU, placeholder addresses stand in for the arrays (no
    launch could reach a device); on a machine with a GPU the same calls run
    with real device buffers in the GPU tests instead."""
    import ctypes
    import torch
    import speculative_decoding_tree_02_gb300 as tv
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: covered with real buffers by the GPU tests")
    for want, call in validation_calls(tv.load_library(), ctypes.c_void_p(256)):
        assert call() == want


def test_product_templates_equal_oracle_templates():
    from oracle import graft as ogr
    from speculative_decoding_tree_02_gb300 import templates
    tp, tr, off = templates.stage_templates()
    otp, otr, ooff = ogr.stage_templates()
    assert np.array_equal(tp, otp) and np.array_equal(tr, otr) and np.array_equal(off, ooff)
    rng = np.random.default_rng(0)
    from synth import random_tree
    pd = random_tree(rng, 25, 8)
    assert np.array_equal(templates.assemble_hybrid(pd, tp[off[1]:off[2]]),
                          ogr.assemble_hybrid(pd, otp[ooff[1]:ooff[2]]))
