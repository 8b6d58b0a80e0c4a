"""CPU checks of the host half of the tree block map (no GPU): the q-major
lists pt_build_blockmap_tree derives on the host from the node intervals
(each q tile's non-empty kv blocks, ascending) equal the oracle's
brute-force block map over every (q, kv) pair, on the workload layouts and
on random trees at several tile shapes.  On the GPU the device classifies
only these tiles, so a tile missing here would lose keys."""
import ctypes

import numpy as np
import pytest

import prefix_tree_block_gb300 as pt
from oracle import oracle as orc
from prefix_tree_block_gb300 import build as ptbuild
from prefix_tree_block_gb300 import workloads as W

SHAPES = [(128, 128), (64, 128), (128, 64), (32, 64), (16, 16)]


@pytest.fixture(scope="module")
def lib():
    ptbuild.build()
    return pt.load_library()


def host_lists(lib, st, BM, BN):
    lengths = np.ascontiguousarray(st.node_lengths, np.int32)
    ptr = np.ascontiguousarray(st.path_ptr, np.int32)
    nodes = np.ascontiguousarray(st.path_nodes, np.int32)
    T = int(lengths.sum())
    nq = -(-T // BM)
    q_ptr = np.zeros(nq + 1, np.int32)
    cap = max(1, nq * (-(-T // BN)))
    kv = np.zeros(cap, np.int32)
    nnz = ctypes.c_int64()
    rc = lib.pt_debug_tree_lists(lengths.ctypes.data, len(lengths), ptr.ctypes.data, nodes.ctypes.data,
                                 len(ptr) - 1, BM, BN, q_ptr.ctypes.data, nq + 1, kv.ctypes.data, cap,
                                 ctypes.byref(nnz))
    assert rc == pt.PT_OK, lib.pt_last_error()
    return q_ptr, kv[:nnz.value]


def check(lib, st, BM, BN):
    q_ptr, kv = host_lists(lib, st, BM, BN)
    want = orc.blockmap(orc.structure_labels(st), BM, BN)
    assert np.array_equal(q_ptr, want["q_ptr"])
    assert np.array_equal(kv, want["kv_idx"])


@pytest.mark.parametrize("c", [1, 2, 4])
def test_workload_layouts(lib, c):
    st = W.config_structure(c)
    check(lib, st, 128, 128)
    if st.T <= 8000:
        check(lib, st, 64, 128)


@pytest.mark.parametrize("BM,BN", SHAPES)
def test_random_trees(lib, BM, BN):
    rng = np.random.default_rng(BM * 1000 + BN)
    for _ in range(12):
        st = W.random_tree(rng, n_nodes=int(rng.integers(1, 14)), max_len=int(rng.integers(1, 300)))
        if st.T == 0:
            continue
        check(lib, st, BM, BN)


def test_grpo_with_empty_prompt_and_one_token_completions(lib):
    st = W.grpo_structure([(0, [1, 1, 130]), (257, [1, 128, 0, 3])])
    for BM, BN in SHAPES:
        check(lib, st, BM, BN)


def test_malformed_tree_rejected(lib):
    lengths = np.array([4, 5], np.int32)
    ptr = np.array([0, 2], np.int32)
    nodes = np.array([1, 0], np.int32)  # a parent with a larger id than its child
    q_ptr = np.zeros(4, np.int32)
    kv = np.zeros(4, np.int32)
    nnz = ctypes.c_int64()
    assert lib.pt_debug_tree_lists(lengths.ctypes.data, 2, ptr.ctypes.data, nodes.ctypes.data, 1, 128, 128,
                                   q_ptr.ctypes.data, 4, kv.ctypes.data, 4, ctypes.byref(nnz)) == pt.PT_ERR_INVALID_ARG
