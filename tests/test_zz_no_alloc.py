"""pt_attn_bwd_noalloc, the backward entry point that allocates nothing.

It exists for callers that cannot call cudaMalloc: a host program that owns
all device memory through its own allocator and gives this library no way to
get scratch, or a latency-critical path where an allocation (which can
synchronise the device) is not allowed.  Its scratch lives in a fixed array
inside the library.  These tests call it through the C ABI (ctypes on
libpt.so) and check that two calls in a row give the same gradients as
pt_attn_bwd with a caller workspace, and the same gradients as the fp64
oracle, within the parity tolerance used for the backward (relative L2 norm
3e-2 for bf16, 1e-5 for fp32).  They also check that on a prepared map the
calls take nothing from the library's device memory pool, and that a
workspace backward on the same map leaves the prepared lists in place.  The
file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import prefix_tree_block_gb300 as pt
from oracle import oracle as orc
from prefix_tree_block_gb300 import workloads as W
from parity import GRAD_RL2, ensure_built, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    return pt.load_library()


def _noalloc(lib, dO, Q, K, V, O, LSE, bm, dtype_code, expect=pt.PT_OK):
    T, Hq, D = Q.shape
    Hkv = K.shape[1]
    dQ, dK, dV = (pt._empty(x.shape, x.dtype, x.device) for x in (Q, K, V))  # guarded in the tests
    rc = lib.pt_attn_bwd_noalloc(dO.data_ptr(), Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(),
                                 LSE.data_ptr(), dtype_code, T, Hq, Hkv, D, 0.0, bm.handle, dQ.data_ptr(),
                                 dK.data_ptr(), dV.data_ptr(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == expect, lib.pt_last_error()
    torch.cuda.synchronize()
    return dQ, dK, dV


def _pool_usage(lib):
    used, reserved = ctypes.c_uint64(), ctypes.c_uint64()
    assert lib.pt_debug_pool_usage(torch.cuda.current_device(), ctypes.byref(used), ctypes.byref(reserved)) == 0
    return used.value, reserved.value


@pytest.mark.parametrize("dtype,D,BM", [("bf16", 64, 128), ("bf16", 128, 128), ("bf16", 256, 128), ("bf16", 512, 128),
                                        ("bf16", 96, 128), ("bf16", 320, 128), ("f32", 32, 16)])
def test_noalloc_matches_workspace_backward_twice(lib, dtype, D, BM):
    st = W.grpo_structure([(300, [100, 41, 250]), (0, [77, 129])])
    q, k, v, do = W.make_tensors(st.T, 4, 2, D, dtype, seed=D)
    Q, K, V, dO = (x.cuda() for x in (q, k, v, do))
    bm = pt.build_blockmap_tree(st.node_lengths, st.path_ptr, st.path_nodes, BM, BM)
    O, LSE = pt.attn_fwd(Q, K, V, bm)
    ref = [x.float().cpu().numpy() for x in pt.attn_bwd(dO, Q, K, V, O, LSE, bm)]
    code = pt.PT_BF16 if dtype == "bf16" else pt.PT_F32
    # a fresh map of the same layout: the workspace backward above may already have built, on bm, the lists
    # the allocation-free call reads (at head_dim 256 they are the same lists)
    bm = pt.build_blockmap_tree(st.node_lengths, st.path_ptr, st.path_nodes, BM, BM)
    if dtype == "bf16" and D in (64, 128, 256, 512):  # the tensor-core path reads per-map work lists: refused until prepared
        _noalloc(lib, dO, Q, K, V, O, LSE, bm, code, expect=pt.PT_ERR_INVALID_ARG)
        assert b"pt_blockmap_prepare_bwd" in lib.pt_last_error()
    elif dtype == "bf16":  # the CUDA-core kernels keep no lists: no preparation needed
        got = [x.float().cpu().numpy() for x in _noalloc(lib, dO, Q, K, V, O, LSE, bm, code)]
        for g, r in zip(got, ref):
            assert rel_l2(g, r) <= GRAD_RL2[dtype]
    bm.prepare_bwd(Q.shape[1], K.shape[1], D)
    bm.prepare_bwd(Q.shape[1], K.shape[1], D)  # idempotent
    torch.cuda.synchronize()
    pool_before = _pool_usage(lib)
    want = orc.attn_bwd(q, k, v, do, orc.structure_labels(st))
    for _ in range(2):
        got = [x.float().cpu().numpy() for x in _noalloc(lib, dO, Q, K, V, O, LSE, bm, code)]
        for g, r, w in zip(got, ref, want):
            assert np.isfinite(g).all()
            assert rel_l2(g, r) <= GRAD_RL2[dtype]
            assert rel_l2(g, w) <= GRAD_RL2[dtype]
    assert _pool_usage(lib) == pool_before  # nothing taken from (or added to) the library's pool
    pt.sync_status()


@pytest.mark.parametrize("D", [64, 128])
def test_noalloc_lists_survive_a_workspace_backward(lib, D):
    """A workspace backward on a prepared map builds lists of its own (long
    columns split across SMs) beside the prepared ones; the allocation-free
    call must still find its lists afterwards."""
    st = W.grpo_structure([(700, [300, 41, 250, 640]), (0, [77, 129])])
    q, k, v, do = W.make_tensors(st.T, 4, 2, D, "bf16", seed=D + 1)
    Q, K, V, dO = (x.cuda() for x in (q, k, v, do))
    bm = pt.build_blockmap_tree(st.node_lengths, st.path_ptr, st.path_nodes)
    O, LSE = pt.attn_fwd(Q, K, V, bm)
    bm.prepare_bwd(4, 2, D)
    first = [x.float().cpu().numpy() for x in _noalloc(lib, dO, Q, K, V, O, LSE, bm, pt.PT_BF16)]
    ws = [x.float().cpu().numpy() for x in pt.attn_bwd(dO, Q, K, V, O, LSE, bm)]
    torch.cuda.synchronize()
    pool_before = _pool_usage(lib)
    again = [x.float().cpu().numpy() for x in _noalloc(lib, dO, Q, K, V, O, LSE, bm, pt.PT_BF16)]
    assert _pool_usage(lib) == pool_before
    want = orc.attn_bwd(q, k, v, do, orc.structure_labels(st))
    for a, b, c, w in zip(first, again, ws, want):
        np.testing.assert_array_equal(a, b)  # the same lists and kernels: bit-identical
        assert rel_l2(a, w) <= GRAD_RL2["bf16"]
        assert rel_l2(c, w) <= GRAD_RL2["bf16"]
    pt.sync_status()


def test_noalloc_head_dim_limits(lib):
    """Head dims as pt_attn_bwd takes them: 1..512; above that unsupported, 0 invalid."""
    st = W.grpo_structure([(40, [9, 20])])
    bm = pt.build_blockmap_tree(st.node_lengths, st.path_ptr, st.path_nodes)
    buf = torch.zeros(st.T * 2 * 520, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(2 * st.T, dtype=torch.float32, device="cuda")
    p = buf.data_ptr()
    for D, want in [(520, pt.PT_ERR_UNSUPPORTED), (0, pt.PT_ERR_INVALID_ARG)]:
        rc = lib.pt_attn_bwd_noalloc(p, p, p, p, p, lse.data_ptr(), pt.PT_BF16, st.T, 2, 1, D, 0.0, bm.handle, p, p,
                                     p, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == want, lib.pt_last_error()
    bm.prepare_bwd(2, 1, 512)  # the largest head dim it takes
    with pytest.raises(pt.PTError) as ei:
        bm.prepare_bwd(2, 1, 520)
    assert ei.value.status == pt.PT_ERR_UNSUPPORTED


def test_noalloc_rejects_shapes_beyond_its_scratch(lib):
    cap = lib.pt_bwd_noalloc_max_scratch_bytes()
    T, Hq = 20000, 64  # needs 2 * 64 * 20096 * 4 bytes, more than the array holds
    assert 2 * Hq * (-(-T // 128) * 128) * 4 > cap
    st = W.docs_structure([T])
    bm = pt.build_blockmap_tree(st.node_lengths, st.path_ptr, st.path_nodes)
    small = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(4, dtype=torch.float32, device="cuda")
    p = small.data_ptr()
    rc = lib.pt_attn_bwd_noalloc(p, p, p, p, p, lse.data_ptr(), pt.PT_BF16, T, Hq, 8, 64, 0.0, bm.handle, p, p, p,
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == pt.PT_ERR_INVALID_ARG
    assert b"scratch" in lib.pt_last_error()
