"""Backward parity: dQ, dK, dV vs the fp64 oracle (relative L2 norm), at
small sizes over all elements and at the workload sizes on sampled rows and
kv columns plus the sum invariants that hold at any size."""
import numpy as np
import pytest

from oracle import oracle as orc
from prefix_tree_block_gb300 import workloads as W
from parity import GRAD_RL2, ensure_built, rel_l2, run_bwd, sample_rows
from test_gpu_fwd import small_structures

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def check_bwd(st, Hq, Hkv, D, dtype, seed, **kw):
    (q, k, v, do), (dQ, dK, dV) = run_bwd(st, Hq, Hkv, D, dtype, seed, **kw)
    wq, wk, wv = orc.attn_bwd(q, k, v, do, orc.structure_labels(st))
    errs = (rel_l2(dQ, wq), rel_l2(dK, wk), rel_l2(dV, wv))
    assert max(errs) <= GRAD_RL2[dtype], errs
    return errs


def test_fp32_workload1():
    cfg = W.CONFIGS[1]
    check_bwd(W.config_structure(1), cfg["Hq"], cfg["Hkv"], cfg["D"], "f32", seed=1, BM=16, BN=16)


@pytest.mark.parametrize("BM,BN", [(16, 16), (32, 64)])
def test_fp32_random_tree(BM, BN):
    rng = np.random.default_rng(77 + BM)
    st = W.random_tree(rng, n_nodes=9, max_len=50)
    check_bwd(st, 4, 2, 40, "f32", seed=4, BM=BM, BN=BN)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("name", ["grpo", "grpo_p0", "tree", "docs"])
def test_tensor_core_bwd_small(D, name):
    check_bwd(small_structures()[name], 4, 2, D, "bf16", seed=D + 1)


@pytest.mark.parametrize("Hq,Hkv", [(1, 1), (8, 1)])
def test_tensor_core_bwd_gqa(Hq, Hkv):
    check_bwd(small_structures()["grpo"], Hq, Hkv, 128, "bf16", seed=Hq + 2)


def test_tensor_core_bwd_dense_map_equal():
    check_bwd(small_structures()["tree"], 2, 1, 64, "bf16", seed=6, dense=True)


@pytest.mark.parametrize("c", [2, 3, 4, 5])
def test_workload_sampled(c):
    cfg = W.CONFIGS[c]
    st = W.config_structure(c)
    Hq, Hkv, D = cfg["Hq"], cfg["Hkv"], cfg["D"]
    (q, k, v, do), (dQ, dK, dV) = run_bwd(st, Hq, Hkv, D, "bf16", seed=c)
    lab = orc.structure_labels(st)
    rows = sample_rows(st, st.T, n_random=24, seed=c)
    wq, _, _ = orc.attn_bwd(q, k, v, do, lab, qrows=rows, want_dkv=False)
    assert rel_l2(dQ[rows], wq) <= GRAD_RL2["bf16"]
    # kv columns: the last token of each node (few rows see it) plus a few
    starts = np.concatenate([[0], np.cumsum(st.node_lengths)[:-1]]).astype(int)
    ends = [int(s + n - 1) for s, n in zip(starts, st.node_lengths) if n > 0]
    rng = np.random.default_rng(c)
    cols = np.array(sorted(set(list(rng.choice(ends, min(8, len(ends)), replace=False)) + [st.T - 1])), np.int64)
    _, wk, wv = orc.attn_bwd(q, k, v, do, lab, kvcols=cols, want_dq=False)
    assert rel_l2(dK[cols], wk) <= GRAD_RL2["bf16"]
    assert rel_l2(dV[cols], wv) <= GRAD_RL2["bf16"]
    # invariants at full size: sum_j dK_j = 0 and sum_j dV_j = sum of dO over
    # rows and the kv head's q heads
    g = Hq // Hkv
    sdo = do.float().numpy().astype(np.float64).reshape(st.T, Hkv, g, D).sum(axis=(0, 2))
    assert rel_l2(dV.sum(axis=0), sdo) <= GRAD_RL2["bf16"]
    scale_k = np.abs(dK).sum(axis=0).max()
    assert np.abs(dK.sum(axis=0)).max() <= 1e-2 * scale_k


@pytest.mark.parametrize("name", ["grpo", "grpo_p0", "tree", "docs"])
def test_head_dim_64_one_pass_and_two_pass(name):
    """At head_dim 64 the workspace picks the backward: with room for the
    fp32 dQ accumulator the one-pass kernel (dQ added up by asynchronous
    reduce-adds), with the two row statistics alone the kv-major and q-major
    kernels.  Both match the oracle and each other, and each launches the
    kernels it should."""
    import prefix_tree_block_gb300 as pt
    import torch

    st = small_structures()[name]
    Hq, Hkv, D = 4, 2, 64
    q, k, v, do = W.make_tensors(st.T, Hq, Hkv, D, "bf16", seed=11)
    Q, K, V, dO = (x.cuda() for x in (q, k, v, do))
    bm = pt.build_blockmap_tree(st.node_lengths, st.path_ptr, st.path_nodes)
    O, LSE = pt.attn_fwd(Q, K, V, bm)
    tpad = -(-st.T // 128) * 128
    stats = 2 * (-(-(4 * tpad * Hq) // 256) * 256)
    full = torch.empty(pt.bwd_workspace_bytes(st.T, Hq, D), dtype=torch.uint8, device="cuda")
    small = torch.empty(stats, dtype=torch.uint8, device="cuda")
    want = orc.attn_bwd(q, k, v, do, orc.structure_labels(st))
    got = {}
    for label, ws in (("one", full), ("two", small)):
        pt.profile_reset()
        pt.profile_enable(True)
        res = pt.attn_bwd(dO, Q, K, V, O, LSE, bm, workspace=ws)
        pt.sync_status()
        n_fused = pt.profile_read("bwd_fused")[0]
        n_dq = pt.profile_read("bwd_dq")[0]
        pt.profile_enable(False)
        assert (n_fused, n_dq) == ((1, 0) if label == "one" else (0, 1))
        got[label] = [x.float().cpu().numpy() for x in res]
        for g, w in zip(got[label], want):
            assert rel_l2(g, w) <= GRAD_RL2["bf16"]
    for a, b in zip(got["one"], got["two"]):
        assert rel_l2(a, b) <= 1e-2
    bm.free()


@pytest.mark.parametrize("Hq,Hkv", [(1, 1), (8, 1), (6, 3)])
def test_head_dim_64_one_pass_gqa(Hq, Hkv):
    """The one-pass head_dim-64 backward over head layouts: MHA, one kv head
    for eight q heads, three groups of two (dK and dV summed over each group's
    q heads inside the kernel, dQ per q head through the accumulator)."""
    check_bwd(small_structures()["grpo"], Hq, Hkv, 64, "bf16", seed=40 + Hq)


def test_head_dim_64_one_pass_without_split_room():
    """A workspace with room for the two statistics and the dQ accumulator
    but none for partial sums: the one-pass kernel runs with no column split
    (every kv-major column one item)."""
    import prefix_tree_block_gb300 as pt
    import torch

    st = W.grpo_structure([(700, [300, 41, 250, 640]), (0, [77, 129])])
    Hq, Hkv, D = 4, 2, 64
    q, k, v, do = W.make_tensors(st.T, Hq, Hkv, D, "bf16", seed=12)
    Q, K, V, dO = (x.cuda() for x in (q, k, v, do))
    bm = pt.build_blockmap_tree(st.node_lengths, st.path_ptr, st.path_nodes)
    O, LSE = pt.attn_fwd(Q, K, V, bm)
    tpad = -(-st.T // 128) * 128
    r256 = lambda n: -(-n // 256) * 256
    need = 2 * r256(4 * tpad * Hq) + r256(4 * tpad * Hq * D)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    pt.profile_reset()
    pt.profile_enable(True)
    res = pt.attn_bwd(dO, Q, K, V, O, LSE, bm, workspace=ws)
    pt.sync_status()
    n_fused = pt.profile_read("bwd_fused")[0]
    n_split = pt.profile_read("bwd_dkdv_finalize")[0]
    pt.profile_enable(False)
    assert n_fused == 1 and n_split == 0
    want = orc.attn_bwd(q, k, v, do, orc.structure_labels(st))
    for g, w in zip((x.float().cpu().numpy() for x in res), want):
        assert rel_l2(g, w) <= GRAD_RL2["bf16"]
    bm.free()


def test_head_dim_64_one_pass_columns_cut_across_ctas():
    """Long prompt columns at a size where the one-pass kernel's work lists
    cut them at each CTA's share of the steps: chunks of one column run on
    consecutive CTAs and write fp32 partial sums that the finalize kernel
    adds.  Every element against the oracle, and against the two-pass
    backward (whose columns stay whole or are cut into equal chunks)."""
    import prefix_tree_block_gb300 as pt
    import torch

    st = W.grpo_structure([(1800, [300, 500, 410, 222]), (600, [200, 77]), (0, [129])])
    Hq, Hkv, D = 8, 2, 64
    q, k, v, do = W.make_tensors(st.T, Hq, Hkv, D, "bf16", seed=13)
    Q, K, V, dO = (x.cuda() for x in (q, k, v, do))
    bm = pt.build_blockmap_tree(st.node_lengths, st.path_ptr, st.path_nodes)
    O, LSE = pt.attn_fwd(Q, K, V, bm)
    tpad = -(-st.T // 128) * 128
    stats = 2 * (-(-(4 * tpad * Hq) // 256) * 256)
    full = torch.empty(pt.bwd_workspace_bytes(st.T, Hq, D), dtype=torch.uint8, device="cuda")
    small = torch.empty(stats, dtype=torch.uint8, device="cuda")
    pt.profile_reset()
    pt.profile_enable(True)
    one = [x.float().cpu().numpy() for x in pt.attn_bwd(dO, Q, K, V, O, LSE, bm, workspace=full)]
    pt.sync_status()
    assert pt.profile_read("bwd_fused")[0] == 1
    pt.profile_enable(False)
    two = [x.float().cpu().numpy() for x in pt.attn_bwd(dO, Q, K, V, O, LSE, bm, workspace=small)]
    want = orc.attn_bwd(q, k, v, do, orc.structure_labels(st))
    for a, b, w in zip(one, two, want):
        assert rel_l2(a, w) <= GRAD_RL2["bf16"]
        assert rel_l2(a, b) <= 1e-2
    bm.free()
