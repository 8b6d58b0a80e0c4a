"""Head dims above 256 (up to 512): forward and backward through the C ABI
against the fp64 oracle.  bf16 at head_dim 512 on a 128 x 128 map runs on
tensor cores (the forward in two passes over the halves of O, the backward in
six passes, one per half of dV, dK and dQ); the other head dims above 256 and
fp32 inputs run on the CUDA-core kernels (fp32 math).  The drafter PR reports FlexAttention failing beyond head_dim 256 on
sm_103, which is why the library takes them at all."""
import numpy as np
import pytest

from oracle import oracle as orc
from prefix_tree_block_gb300 import workloads as W
from parity import FWD_ATOL, GRAD_RL2, LSE_ATOL, ensure_built, rel_l2, run_bwd, run_fwd, sample_rows
from test_gpu_bwd import check_bwd
from test_gpu_fwd import check_fwd, small_structures

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


@pytest.mark.parametrize("D", [264, 320, 512])
@pytest.mark.parametrize("name", ["grpo_p0", "tree", "docs"])
def test_bf16_fwd_bwd(D, name):
    st = small_structures()[name]
    check_fwd(st, 4, 2, D, "bf16", seed=D)
    check_bwd(st, 4, 2, D, "bf16", seed=D + 1)


@pytest.mark.parametrize("name", ["grpo", "grpo_p0", "tree", "docs"])
@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (3, 3), (8, 1)])
def test_tensor_core_fwd_head_dim_512(name, Hq, Hkv):
    """Every element of O and LSE at head_dim 512 (tensor cores) on layouts
    with ragged tails, an empty prompt and one-token completions."""
    check_fwd(small_structures()[name], Hq, Hkv, 512, "bf16", seed=Hq * 7 + Hkv)


def test_tensor_core_fwd_head_dim_512_dense_map():
    check_fwd(small_structures()["tree"], 2, 1, 512, "bf16", seed=11, dense=True)


@pytest.mark.parametrize("name", ["grpo", "grpo_p0", "tree", "docs"])
@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (3, 3), (8, 1)])
def test_tensor_core_bwd_head_dim_512(name, Hq, Hkv):
    """Every element of dQ, dK, dV at head_dim 512 (tensor cores), relative L2."""
    check_bwd(small_structures()[name], Hq, Hkv, 512, "bf16", seed=Hq * 5 + Hkv)


def test_tensor_core_bwd_head_dim_512_dense_map():
    check_bwd(small_structures()["tree"], 2, 1, 512, "bf16", seed=12, dense=True)


@pytest.mark.parametrize("BM,BN", [(128, 128), (32, 64)])
def test_fp32_fwd_bwd(BM, BN):
    rng = np.random.default_rng(BM + 5)
    st = W.random_tree(rng, n_nodes=8, max_len=60)
    check_fwd(st, 2, 1, 384, "f32", seed=3, BM=BM, BN=BN)
    check_bwd(st, 2, 1, 384, "f32", seed=4, BM=BM, BN=BN)


def test_workload_sampled():
    """Workload 7 (packed documents at head_dim 512) at full size, sampled
    rows and kv columns, plus the gradient sums that hold at any size."""
    cfg = W.CONFIGS[7]
    st = W.config_structure(7)
    Hq, Hkv, D = cfg["Hq"], cfg["Hkv"], cfg["D"]
    (q, k, v), O, L = run_fwd(st, Hq, Hkv, D, "bf16", seed=7)
    lab = orc.structure_labels(st)
    rows = sample_rows(st, st.T, n_random=24, seed=7)
    Ow, Lw = orc.attn_fwd(q, k, v, lab, rows=rows)
    assert np.abs(O[rows] - Ow).max() <= FWD_ATOL["bf16"]
    assert np.abs(L[:, rows] - Lw).max() <= LSE_ATOL["bf16"]
    (q, k, v, do), (dQ, dK, dV) = run_bwd(st, Hq, Hkv, D, "bf16", seed=7)
    wq, _, _ = orc.attn_bwd(q, k, v, do, lab, qrows=rows, want_dkv=False)
    assert rel_l2(dQ[rows], wq) <= GRAD_RL2["bf16"]
    cols = np.array(sorted(set(int(x) for x in rows)), np.int64)
    _, wk, wv = orc.attn_bwd(q, k, v, do, lab, kvcols=cols, want_dq=False)
    assert rel_l2(dK[cols], wk) <= GRAD_RL2["bf16"]
    assert rel_l2(dV[cols], wv) <= GRAD_RL2["bf16"]
    g = Hq // Hkv
    sdo = do.float().numpy().astype(np.float64).reshape(st.T, Hkv, g, D).sum(axis=(0, 2))
    assert rel_l2(dV.sum(axis=0), sdo) <= GRAD_RL2["bf16"]
    assert np.abs(dK.sum(axis=0)).max() <= 1e-2 * np.abs(dK).sum(axis=0).max()
