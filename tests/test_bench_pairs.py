"""The benchmark's useful-pair counts (its flop numerator) against the oracle's
keep matrices: draft-block layouts and trees."""
import numpy as np
import pytest

import bench
from oracle import draft as OD
from oracle import oracle as OR
from prefix_tree_block_gb300 import workloads as W


@pytest.mark.parametrize("seed", range(5))
def test_draft_pairs_match_mask(seed):
    rng = np.random.default_rng(seed)
    st = W.draft_structure(rng, int(rng.integers(60, 300)), 20, 90, int(rng.integers(2, 9)), int(rng.choice([2, 4, 8])),
                           causal=bool(seed % 2), window=int(rng.integers(5, 40)) if seed % 3 == 0 else 0)
    if seed == 4:
        st.block_keep = rng.random(st.anchors.size) > 0.3
    assert bench.draft_pairs(st) == int(OD.draft_mask(**st.kwargs()).sum())


@pytest.mark.parametrize("c", [1, 4])
def test_tree_pairs_match_oracle(c):
    st = W.config_structure(c)
    assert bench.useful_pairs(st) == OR.count_pairs(OR.structure_labels(st))


def test_draft_workload_anchors_keep_blocks_in_document():
    st = W.config_structure(6)
    ends = np.cumsum(np.bincount(st.ctx_doc))
    assert np.all(st.anchors + st.block_size <= ends[st.anchor_doc])
    assert np.all(st.ctx_doc[st.anchors] == st.anchor_doc)


@pytest.mark.parametrize("c", [1, 4])
def test_dense_keep_mask_matches_oracle(c):
    """The [T, T] mask the bench hands to torch SDPA (its secondary comparison) is the oracle's keep matrix."""
    st = W.config_structure(c)
    got = bench.dense_keep_mask(st, "cpu").numpy()
    np.testing.assert_array_equal(got, OR.dense_mask(OR.structure_labels(st)).astype(bool))


@pytest.mark.parametrize("seed", range(4))
def test_dense_keep_mask_random_trees(seed):
    rng = np.random.default_rng(70 + seed)
    st = W.random_tree(rng, n_nodes=int(rng.integers(1, 25)), max_len=int(rng.integers(1, 60)))
    got = bench.dense_keep_mask(st, "cpu").numpy()
    np.testing.assert_array_equal(got, OR.dense_mask(OR.structure_labels(st)).astype(bool))
