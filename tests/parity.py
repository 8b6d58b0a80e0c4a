"""Shared helpers for the GPU parity tests: run the library through its
binding and compare with the fp64 oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import prefix_tree_block_gb300 as pt
from oracle import oracle as orc
from prefix_tree_block_gb300 import workloads as W

# Tolerances: forward max-abs 2e-2 (bf16) / 1e-5 (fp32); gradients relative
# L2 3e-2 (bf16) / 1e-5 (fp32); block map bit-exact.
FWD_ATOL = {"bf16": 2e-2, "f32": 1e-5}
GRAD_RL2 = {"bf16": 3e-2, "f32": 1e-5}
LSE_ATOL = {"bf16": 2e-3, "f32": 1e-5}


def ensure_built():
    from prefix_tree_block_gb300 import build as b

    b.build()
    pt.load_library()


def to_dev(x):
    return x.contiguous().cuda()


def gpu_blockmap(st, BM=128, BN=128, form="tree"):
    if form == "tree":
        return pt.build_blockmap_tree(st.node_lengths, st.path_ptr, st.path_nodes, BM, BN)
    g = torch.as_tensor(st.group_id, dtype=torch.int32).cuda()
    s = torch.as_tensor(st.suffix_id, dtype=torch.int32).cuda()
    return pt.build_blockmap_seg(g, s, BM, BN)


def compare_blockmap(got: dict, want: dict):
    for k in ("q_ptr", "kv_idx", "kind", "k_ptr", "q_idx", "kindT"):
        np.testing.assert_array_equal(got[k], want[k], err_msg=k)
    assert got["nnz"] == want["nnz"]


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b.ravel())
    return float(np.linalg.norm((a - b).ravel()) / max(den, 1e-300))


def sample_rows(st, T, n_random=48, seed=0):
    """Rows that stress the layout: ends, tile edges, node starts and ends,
    plus a seeded random sample."""
    rng = np.random.default_rng(seed)
    starts = np.concatenate([[0], np.cumsum(st.node_lengths)[:-1]]).astype(int)
    cand = {0, T - 1, 127, 128, T // 2}
    for s, n in zip(starts, st.node_lengths):
        if n > 0:
            cand.update({int(s), int(s + n - 1)})
    cand = sorted(c for c in cand if 0 <= c < T)
    if len(cand) > 64:
        cand = list(rng.choice(cand, 64, replace=False))
    cand += list(rng.integers(0, T, n_random))
    return np.array(sorted(set(int(c) for c in cand)), np.int64)


def run_fwd(st, Hq, Hkv, D, dtype, seed, BM=128, BN=128, form="tree", dense=False):
    q, k, v, _ = W.make_tensors(st.T, Hq, Hkv, D, dtype, seed)
    bm = gpu_blockmap(st, BM, BN, form)
    if dense:
        bm = bm.dense()
    O, L = pt.attn_fwd(to_dev(q), to_dev(k), to_dev(v), bm)
    pt.sync_status()
    return (q, k, v), O.float().cpu().numpy(), L.cpu().numpy()


def run_bwd(st, Hq, Hkv, D, dtype, seed, BM=128, BN=128, dense=False):
    q, k, v, do = W.make_tensors(st.T, Hq, Hkv, D, dtype, seed)
    bm = gpu_blockmap(st, BM, BN)
    if dense:
        bm = bm.dense()
    Q, K, V, dO = (to_dev(x) for x in (q, k, v, do))
    O, L = pt.attn_fwd(Q, K, V, bm)
    dQ, dK, dV = pt.attn_bwd(dO, Q, K, V, O, L, bm)
    pt.sync_status()
    return (q, k, v, do), tuple(x.float().cpu().numpy() for x in (dQ, dK, dV))
