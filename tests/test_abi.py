"""CPU checks of the C-ABI library: it builds, loads, exports every symbol
include/pt.h declares, and rejects malformed inputs on the host before any
launch (no GPU needed for any of these)."""
import ctypes
import os
import re

import numpy as np
import pytest

import prefix_tree_block_gb300 as pt
from prefix_tree_block_gb300 import build as ptbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    ptbuild.build()
    return pt.load_library()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "pt.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pt_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_path():
    syms = declared_symbols()
    for s in ("pt_build_blockmap_tree", "pt_build_blockmap_seg", "pt_attn_fwd", "pt_attn_bwd"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert not missing, missing


def test_workspace_size(lib):
    T, Hq, D = 1000, 14, 64
    n = pt.bwd_workspace_bytes(T, Hq, D)
    tpad = -(-T // 128) * 128
    assert n >= 2 * 4 * tpad * Hq  # Delta and LSE*log2(e), [Hq, Tpad] fp32 each
    assert n % 256 == 0


@pytest.mark.parametrize("lengths,paths", [
    ([2, 2], [[1, 0]]),                  # child before parent
    ([2, 2, 2], [[0, 1], [0, 2], [1, 2]]),  # two parents
    ([2, 2, 2], [[0, 1]]),               # node on no path
    ([2, -1], [[0, 1]]),                 # negative length
    ([2, 2], [[0, 9]]),                  # node out of range
])
def test_invalid_tree_rejected_on_host(lib, lengths, paths):
    ptr = np.cumsum([0] + [len(p) for p in paths]).astype(np.int32)
    nodes = np.array([n for p in paths for n in p], np.int32)
    with pytest.raises(pt.PTError) as ei:
        pt.build_blockmap_tree(lengths, ptr, nodes, stream=_null_stream())
    assert ei.value.status == pt.PT_ERR_INVALID_ARG
    assert lib.pt_last_error()


def test_null_map_rejected(lib):
    rc = lib.pt_attn_fwd(None, None, None, 0, 10, 2, 2, 64, 0.0, None, None, None, None)
    assert rc == pt.PT_ERR_INVALID_ARG
    assert b"block map" in lib.pt_last_error()


def test_null_out_rejected(lib):
    nl = np.array([4], np.int32)
    pp = np.array([0, 1], np.int32)
    pn = np.array([0], np.int32)
    rc = lib.pt_build_blockmap_tree(nl.ctypes.data, 1, pp.ctypes.data, pn.ctypes.data, 1, 128, 128, None, None)
    assert rc == pt.PT_ERR_INVALID_ARG


class _S:
    cuda_stream = 0


def _null_stream():
    return _S()


def test_host_checks_before_any_device_work(lib):
    """Argument checks that return before any CUDA call, so they run without a GPU."""
    h = ctypes.c_void_p()
    assert lib.pt_hoststep_create(pt.PT_BF16, 100, 4, 2, 520, ctypes.byref(h)) == pt.PT_ERR_UNSUPPORTED
    assert b"head_dim" in lib.pt_last_error()
    assert lib.pt_hoststep_create(pt.PT_BF16, 100, 4, 2, 100, ctypes.byref(h)) == pt.PT_ERR_UNSUPPORTED
    assert lib.pt_hoststep_create(pt.PT_BF16, 100, 4, 3, 64, ctypes.byref(h)) == pt.PT_ERR_INVALID_ARG
    assert lib.pt_hoststep_create(pt.PT_F32, 100, 4, 2, 0, ctypes.byref(h)) == pt.PT_ERR_INVALID_ARG
    assert not h.value
    rc = lib.pt_attn_bwd_noalloc(None, None, None, None, None, None, pt.PT_BF16, 10, 2, 2, 64, 0.0, None, None, None,
                                 None, None)
    assert rc == pt.PT_ERR_INVALID_ARG and b"NULL" in lib.pt_last_error()
    assert lib.pt_blockmap_prepare_bwd(None, 2, 2, 64, None) == pt.PT_ERR_INVALID_ARG
