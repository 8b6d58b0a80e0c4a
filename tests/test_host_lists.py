"""CPU checks of the host half of the tree and draft-block maps (no GPU): the
q-major lists pt_build_blockmap_tree derives on the host from the node
intervals, and pt_build_blockmap_draft from the blocks' ranges (each q
tile's non-empty kv blocks, ascending), equal the oracle's brute-force block
maps over every (q, kv) pair, on the workload layouts and on random layouts;
the draft build's closed-form kept-pair count equals the oracle mask's.  On
the GPU the device classifies only these tiles, so a tile missing here would
lose keys."""
import ctypes

import numpy as np
import pytest

import prefix_tree_block_gb300 as pt
from oracle import draft as OD
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


def draft_layout(seed):
    """Seeded draft layout: context, anchors, block size, dropped blocks,
    causal or not, a window or documents."""
    rng = np.random.default_rng(1000 + seed)
    S = int(rng.integers(100, 900))
    bs = int(rng.choice([1, 4, 8, 16, 24]))
    nb = int(rng.integers(1, 40))
    anchors = np.sort(rng.integers(0, S + 1, nb)).astype(np.int32)
    keep = (rng.random(nb) > 0.15).astype(np.uint8)
    causal = bool(seed % 2)
    window = int(rng.integers(1, 300)) if seed % 3 == 1 else 0
    ctx_doc = anchor_doc = None
    if seed % 3 == 2:
        cuts = np.sort(rng.choice(np.arange(1, S), 3, replace=False))
        ctx_doc = np.searchsorted(cuts, np.arange(S), side="right").astype(np.int32)
        anchor_doc = ctx_doc[np.maximum(anchors - 1, 0)].astype(np.int32)
        anchor_doc[rng.random(nb) < 0.1] = 99  # an anchor whose document is not in the context
    return dict(ctx_len=S, anchors=anchors, block_size=bs, block_keep=keep, causal=causal, window=window,
                ctx_doc=ctx_doc, anchor_doc=anchor_doc)


def draft_lists(lib, lay):
    anchors = np.ascontiguousarray(lay["anchors"], np.int32)
    keep = np.ascontiguousarray(lay["block_keep"], np.uint8)
    T = lay["ctx_len"] + len(anchors) * lay["block_size"]
    nq = -(-T // 128)
    q_ptr = np.zeros(nq + 1, np.int32)
    cap = max(1, nq * nq)
    kv = np.zeros(cap, np.int32)
    nnz, pairs = ctypes.c_int64(), ctypes.c_int64()
    cd = None if lay["ctx_doc"] is None else np.ascontiguousarray(lay["ctx_doc"], np.int32)
    ad = None if lay["anchor_doc"] is None else np.ascontiguousarray(lay["anchor_doc"], np.int32)
    rc = lib.pt_debug_draft_lists(lay["ctx_len"], len(anchors), lay["block_size"], anchors.ctypes.data,
                                  keep.ctypes.data, int(lay["causal"]), lay["window"],
                                  None if cd is None else cd.ctypes.data, None if ad is None else ad.ctypes.data,
                                  q_ptr.ctypes.data, nq + 1, kv.ctypes.data, cap, ctypes.byref(nnz),
                                  ctypes.byref(pairs))
    assert rc == pt.PT_OK, lib.pt_last_error()
    return q_ptr, kv[:nnz.value], pairs.value


@pytest.mark.parametrize("seed", range(12))
def test_draft_lists_and_kept_pairs(lib, seed):
    lay = draft_layout(seed)
    mask = OD.draft_mask(**lay)
    want = OD.mask_blockmap(mask, 128, 128)
    q_ptr, kv, pairs = draft_lists(lib, lay)
    assert np.array_equal(q_ptr, want["q_ptr"])
    assert np.array_equal(kv, want["kv_idx"])
    assert pairs == int(mask.sum(dtype=np.int64))


def test_draft_bad_layout_rejected(lib):
    anchors = np.array([11], np.int32)  # beyond the context
    q_ptr = np.zeros(4, np.int32)
    kv = np.zeros(4, np.int32)
    nnz, pairs = ctypes.c_int64(), ctypes.c_int64()
    assert lib.pt_debug_draft_lists(10, 1, 4, anchors.ctypes.data, None, 0, 0, None, None, q_ptr.ctypes.data, 4,
                                    kv.ctypes.data, 4, ctypes.byref(nnz), ctypes.byref(pairs)) == pt.PT_ERR_INVALID_ARG
