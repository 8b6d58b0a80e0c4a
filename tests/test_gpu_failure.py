"""Failure reporting on the GPU without faulting it: a kernel waits on a
barrier nothing completes, the bounded wait gives up after about a second,
the status word reports PT_ERR_TIMEOUT, and the context keeps working."""
import ctypes

import numpy as np
import pytest
import torch

import prefix_tree_block_gb300 as pt
from oracle import oracle as orc
from prefix_tree_block_gb300 import workloads as W
from parity import FWD_ATOL, ensure_built, run_fwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def test_bounded_wait_times_out_and_context_survives():
    lib = pt.load_library()
    pt.sync_status()  # start clean
    s = torch.cuda.current_stream()
    assert lib.pt_debug_wait_timeout(ctypes.c_void_p(s.cuda_stream)) == pt.PT_OK
    with pytest.raises(pt.PTError) as ei:
        pt.sync_status()
    assert ei.value.status == pt.PT_ERR_TIMEOUT
    pt.sync_status()  # the status word was cleared
    st = W.grpo_structure([(150, [60, 130])])
    (q, k, v), O, _ = run_fwd(st, 2, 1, 64, "bf16", seed=3)
    Ow, _ = orc.attn_fwd(q, k, v, orc.structure_labels(st))
    assert np.abs(O - Ow).max() <= FWD_ATOL["bf16"]


def test_invalid_calls_fail_before_launch():
    st = W.grpo_structure([(100, [30])])
    bm = pt.build_blockmap_tree(st.node_lengths, st.path_ptr, st.path_nodes)
    q, k, v, _ = W.make_tensors(st.T, 2, 1, 64, "bf16", 1)
    Q, K, V = q.cuda(), k.cuda(), v.cuda()
    n0 = pt.launch_count()
    with pytest.raises(pt.PTError) as ei:  # head counts that do not divide
        pt.attn_fwd(Q, K.repeat(1, 3, 1).contiguous()[:, :3], V.repeat(1, 3, 1).contiguous()[:, :3], bm)
    assert ei.value.status == pt.PT_ERR_INVALID_ARG
    with pytest.raises(pt.PTError) as ei:  # wrong T for the map
        pt.attn_fwd(Q[:-1].contiguous(), K[:-1].contiguous(), V[:-1].contiguous(), bm)
    assert ei.value.status == pt.PT_ERR_INVALID_ARG
    assert pt.launch_count() == n0
