"""Forward parity: the library's O and LSE vs the fp64 oracle on the same
seeded inputs (element by element at small sizes; sampled rows at the full
workload sizes)."""
import numpy as np
import pytest

from oracle import oracle as orc
from prefix_tree_block_gb300 import workloads as W
from parity import FWD_ATOL, LSE_ATOL, ensure_built, run_fwd, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def small_structures():
    rng = np.random.default_rng(11)
    return {
        "grpo": W.grpo_structure([(int(rng.integers(100, 400)), [int(x) for x in rng.integers(30, 200, 4)])
                                  for _ in range(2)]),
        "grpo_p0": W.grpo_structure([(0, [70, 300, 5]), (129, [1, 127])]),
        "tree": W.tree_structure([200, 90, 60, 150, 40, 77, 3],
                                 [[0, 1, 2], [0, 1, 3], [0, 4, 5], [0, 4, 6]]),
        "docs": W.docs_structure([64, 700, 33, 1, 250]),
    }


def check_fwd(st, Hq, Hkv, D, dtype, seed, **kw):
    (q, k, v), O, L = run_fwd(st, Hq, Hkv, D, dtype, seed, **kw)
    Ow, Lw = orc.attn_fwd(q, k, v, orc.structure_labels(st))
    err = np.abs(O - Ow).max()
    lerr = np.abs(L - Lw).max()
    assert err <= FWD_ATOL[dtype], f"O max-abs {err}"
    assert lerr <= LSE_ATOL[dtype], f"LSE max-abs {lerr}"
    return err


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("name", ["grpo", "grpo_p0", "tree", "docs"])
def test_tensor_core_fwd_small(D, name):
    st = small_structures()[name]
    check_fwd(st, 4, 2, D, "bf16", seed=D)


@pytest.mark.parametrize("Hq,Hkv", [(1, 1), (8, 1), (6, 3)])
def test_tensor_core_fwd_gqa(Hq, Hkv):
    check_fwd(small_structures()["grpo"], Hq, Hkv, 128, "bf16", seed=Hq)


def test_tensor_core_fwd_dense_map_equal():
    st = small_structures()["tree"]
    check_fwd(st, 2, 1, 128, "bf16", seed=5, dense=True)


def test_tensor_core_fwd_seg_form():
    st = small_structures()["grpo"]
    check_fwd(st, 2, 2, 64, "bf16", seed=3, form="seg")


def test_fp32_workload1():
    st = W.config_structure(1)
    cfg = W.CONFIGS[1]
    check_fwd(st, cfg["Hq"], cfg["Hkv"], cfg["D"], "f32", seed=1, BM=16, BN=16)


@pytest.mark.parametrize("BM,BN", [(16, 16), (128, 128), (32, 64)])
def test_fp32_random_tree(BM, BN):
    rng = np.random.default_rng(BM + BN)
    st = W.random_tree(rng, n_nodes=10, max_len=60)
    check_fwd(st, 4, 2, 48, "f32", seed=2, BM=BM, BN=BN)


def test_bf16_cuda_core_head_dim():
    # head_dim 32 is served by the CUDA-core kernel
    check_fwd(small_structures()["docs"], 2, 1, 32, "bf16", seed=9)


@pytest.mark.parametrize("c", [2, 3, 4, 5])
def test_workload_sampled_rows(c):
    cfg = W.CONFIGS[c]
    st = W.config_structure(c)
    (q, k, v), O, L = run_fwd(st, cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["dtype"], seed=c)
    rows = sample_rows(st, st.T, seed=c)
    Ow, Lw = orc.attn_fwd(q, k, v, orc.structure_labels(st), rows=rows)
    assert np.abs(O[rows] - Ow).max() <= FWD_ATOL["bf16"]
    assert np.abs(L[:, rows] - Lw).max() <= LSE_ATOL["bf16"]
    assert np.isfinite(O).all() and np.isfinite(L).all()
