"""Block map on the GPU vs the oracle's brute-force map: bit-exact."""
import numpy as np
import pytest
import torch

import prefix_tree_block_gb300 as pt
from oracle import oracle as orc
from prefix_tree_block_gb300 import workloads as W
from parity import compare_blockmap, ensure_built, gpu_blockmap

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


@pytest.mark.parametrize("c", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("form", ["tree", "seg"])
def test_workload_blockmaps(c, form):
    st = W.config_structure(c)
    if form == "seg" and st.group_id is None:
        pytest.skip("depth-3 tree has no segment form")
    BM = BN = 16 if c == 1 else 128
    got = gpu_blockmap(st, BM, BN, form)
    want = orc.blockmap(orc.structure_labels(st), BM, BN)
    compare_blockmap(got.export(), want)
    assert got.n_full == int((want["kind"] == 1).sum())


@pytest.mark.parametrize("seed", range(12))
def test_random_trees(seed):
    rng = np.random.default_rng(500 + seed)
    st = W.random_tree(rng, n_nodes=int(rng.integers(1, 30)), max_len=int(rng.integers(1, 300)))
    if st.T == 0:
        pytest.skip("empty")
    BM, BN = [(128, 128), (16, 16), (64, 32), (32, 128)][seed % 4]
    want = orc.blockmap(orc.structure_labels(st), BM, BN)
    compare_blockmap(gpu_blockmap(st, BM, BN).export(), want)


@pytest.mark.parametrize("seed", range(6))
def test_random_grpo_seg_form(seed):
    rng = np.random.default_rng(900 + seed)
    specs = [(int(rng.integers(0, 400)), [int(x) for x in rng.integers(1, 300, int(rng.integers(1, 6)))])
             for _ in range(int(rng.integers(1, 4)))]
    st = W.grpo_structure(specs)
    want = orc.blockmap(orc.seg_labels(st.group_id, st.suffix_id), 128, 128)
    compare_blockmap(gpu_blockmap(st, 128, 128, "seg").export(), want)


@pytest.mark.parametrize("g,s", [
    ([0, 0, 0, 0], [1, 1, -1, -1]),
    ([0, 0, 1, 1, 0], [-1, -1, -1, -1, -1]),
    ([0, 0, 0, 1, 1], [-1, 3, 3, 4, 3]),
    ([0, 0, 0], [-1, 2, -1]),
    ([0, 7, 7], [-1, -1, -1]),  # group id out of [0, T)
])
def test_invalid_segments_rejected(g, s):
    with pytest.raises(pt.PTError) as ei:
        pt.build_blockmap_seg(torch.tensor(g, dtype=torch.int32).cuda(), torch.tensor(s, dtype=torch.int32).cuda())
    assert ei.value.status == pt.PT_ERR_INVALID_ARG


def test_dense_map_lists_every_tile():
    st = W.grpo_structure([(300, [100, 50])])
    d = gpu_blockmap(st).dense().export()
    nq = nk = -(-st.T // 128)
    assert d["nnz"] == nq * nk
    assert (d["kind"] == 2).all()
    np.testing.assert_array_equal(d["q_ptr"], np.arange(nq + 1) * nk)


def test_empty_layout():
    st = W.grpo_structure([(0, [0])])
    bm = gpu_blockmap(st)
    assert bm.T == 0 and bm.nnz == 0


def unpack_bits(words):
    """[n, 128, 4] uint32 -> [n, 128, 128] bool (bit b of word w = column 32w + b)."""
    w = np.asarray(words, np.uint32)
    bits = (w[..., None] >> np.arange(32, dtype=np.uint32)) & 1
    return bits.reshape(w.shape[0], 128, 128).astype(bool)


@pytest.mark.parametrize("case", ["c2", "tree", "ragged", "dense"])
def test_tile_masks_bit_exact(case):
    rng = np.random.default_rng(31)
    st = {"c2": lambda: W.config_structure(2),
          "tree": lambda: W.config_structure(4),
          "ragged": lambda: W.random_tree(rng, n_nodes=17, max_len=200),
          "dense": lambda: W.grpo_structure([(150, [90, 33]), (0, [200])])}[case]()
    bm = gpu_blockmap(st)
    if case == "dense":
        bm = bm.dense()
    lst = bm.export()
    mk = bm.export_masks()
    dense = orc.dense_mask(orc.structure_labels(st)).astype(bool)
    T = st.T
    pad = np.zeros((bm.nq * 128, bm.nk * 128), bool)
    pad[:T, :T] = dense
    rows, cols = unpack_bits(mk["mask_rows"]), unpack_bits(mk["mask_cols"])
    seen = set()
    for i in range(bm.nq):
        for e in range(lst["q_ptr"][i], lst["q_ptr"][i + 1]):
            j, kind, s = lst["kv_idx"][e], lst["kind"][e], mk["pidx"][e]
            want = pad[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
            if kind == 1:
                assert s == -1 and want.all()
                continue
            assert s >= 0 and s not in seen
            seen.add(s)
            np.testing.assert_array_equal(rows[s], want)
            np.testing.assert_array_equal(cols[s], want.T)
    assert len(seen) == bm.nnz - bm.n_full
    # the kv-major list points at the same slots
    for j in range(bm.nk):
        for e in range(lst["k_ptr"][j], lst["k_ptr"][j + 1]):
            i, s = lst["q_idx"][e], mk["pidxT"][e]
            row_e = lst["q_ptr"][i] + np.searchsorted(lst["kv_idx"][lst["q_ptr"][i]:lst["q_ptr"][i + 1]], j)
            assert s == mk["pidx"][row_e]


def test_empty_layout_attention_and_host_lists():
    """T = 0 through the forward and backward (nothing launched, nothing to compare), and a tree whose
    first sample holds only zero-length nodes: its lists, built on the host, must match the oracle."""
    st = W.grpo_structure([(0, [0])])
    bm = gpu_blockmap(st)
    Q = torch.empty(0, 2, 64, dtype=torch.bfloat16, device="cuda")
    K = torch.empty(0, 1, 64, dtype=torch.bfloat16, device="cuda")
    O, L = pt.attn_fwd(Q, K, K, bm)
    dQ, dK, dV = pt.attn_bwd(Q, Q, K, K, O, L, bm)
    assert O.numel() == 0 and dQ.numel() == 0 and dK.numel() == 0
    pt.sync_status()
    st = W.tree_structure([0, 0, 130, 0, 300], [[0, 1], [0, 2], [0, 3, 4]])
    compare_blockmap(gpu_blockmap(st).export(), orc.blockmap(orc.structure_labels(st), 128, 128))


@pytest.mark.parametrize("c", [2, 4])
def test_tile_missing_from_host_lists_is_caught_on_device(c):
    """For a tree at 128 x 128 tiles the host builds the lists and the device
    only classifies the listed tiles.  The device sums the kept pairs over
    them and checks the sum against the tree's closed-form count, so a
    non-empty tile dropped from the host's lists (the test hook drops one)
    shows up as PT_ERR_INVALID_ARG at the next sync; the next build is clean."""
    lib = pt.load_library()
    st = W.config_structure(c)
    lib.pt_debug_drop_listed_tile(1)
    try:
        bm = pt.build_blockmap_tree(st.node_lengths, st.path_ptr, st.path_nodes, 128, 128)
        with pytest.raises(pt.PTError) as ei:
            pt.sync_status()
        assert ei.value.status == pt.PT_ERR_INVALID_ARG
        assert bm.nnz == orc.blockmap(orc.structure_labels(st), 128, 128)["nnz"] - 1
        bm.free()
    finally:
        lib.pt_debug_drop_listed_tile(0)
    bm = pt.build_blockmap_tree(st.node_lengths, st.path_ptr, st.path_nodes, 128, 128)
    pt.sync_status()
    compare_blockmap(bm.export(), orc.blockmap(orc.structure_labels(st), 128, 128))
    bm.free()
