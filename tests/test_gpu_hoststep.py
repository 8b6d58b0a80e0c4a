"""Forward and backward from host memory (pt_hoststep): every pipelined step's
host gradients equal the device-resident path's on the same inputs and the
fp64 oracle's, and the last step's forward outputs (O, LSE) equal the
oracle's."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import prefix_tree_block_gb300 as pt
from oracle import oracle as orc
from prefix_tree_block_gb300 import workloads as W
from parity import FWD_ATOL, GRAD_RL2, LSE_ATOL, rel_l2

pytestmark = pytest.mark.gpu


def _device_grads(q, k, v, do, st):
    Q, K, V, dO = (x.cuda() for x in (q, k, v, do))
    bm = pt.build_blockmap_tree(st.node_lengths, st.path_ptr, st.path_nodes)
    O, L = pt.attn_fwd(Q, K, V, bm)
    dQ, dK, dV = pt.attn_bwd(dO, Q, K, V, O, L, bm)
    torch.cuda.synchronize()
    bm.free()
    return dQ.cpu(), dK.cpu(), dV.cpu()


@pytest.mark.parametrize("workload", [2])
def test_hoststep_pipeline_matches_device_path(workload):
    cfg = W.CONFIGS[workload]
    st = W.config_structure(workload)
    Hq, Hkv, D = cfg["Hq"], cfg["Hkv"], cfg["D"]
    # three steps with different inputs, each into its own host outputs, so a
    # buffer set reused too early would show up as another step's gradients
    steps = []
    for i in range(3):
        q, k, v, do = W.make_tensors(st.T, Hq, Hkv, D, "bf16", 100 + i)
        steps.append(tuple(x.pin_memory() for x in (q, k, v, do)))
    outs = [tuple(torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in (s[0], s[1], s[2])) for s in steps]
    hs = pt.HostStep(torch.bfloat16, st.T, Hq, Hkv, D)
    maps = []
    for (q, k, v, do), (dq, dk, dv) in zip(steps, outs):
        bm = pt.build_blockmap_tree(st.node_lengths, st.path_ptr, st.path_nodes)
        hs.run(q, k, v, do, bm, dq, dk, dv)
        maps.append(bm)
    hs.sync()
    torch.cuda.synchronize()
    pt.sync_status()
    O_last, L_last = hs.last_forward()
    for bm in maps:
        bm.free()
    hs.free()
    lab = orc.structure_labels(st)
    q, k, v, do = steps[-1]
    Ow, Lw = orc.attn_fwd(q, k, v, lab)
    assert np.abs(O_last.float().numpy() - Ow).max() <= FWD_ATOL["bf16"]
    assert np.abs(L_last.numpy() - Lw).max() <= LSE_ATOL["bf16"]
    for (q, k, v, do), (dq, dk, dv) in zip(steps, outs):
        rq, rk, rv = _device_grads(q, k, v, do, st)
        want = orc.attn_bwd(q, k, v, do, lab)
        for got, ref, w in zip((dq, dk, dv), (rq, rk, rv), want):
            g, r = got.float().numpy(), ref.float().numpy()
            # same kernels on the same inputs: equal up to the order of fp32
            # partial sums of split columns
            assert np.linalg.norm(g - r) <= 1e-3 * np.linalg.norm(r) + 1e-6
            assert rel_l2(g, w) <= GRAD_RL2["bf16"]


def test_hoststep_rejects_bad_arguments():
    with pytest.raises(pt.PTError):
        pt.HostStep(torch.bfloat16, 256, 3, 2, 64)  # Hq not a multiple of Hkv
    hs = pt.HostStep(torch.bfloat16, 256, 2, 1, 64)
    st = W.config_structure(1)
    bm = pt.build_blockmap_tree(st.node_lengths, st.path_ptr, st.path_nodes)  # T = 48, not 256
    x = torch.zeros(256, 2, 64, dtype=torch.bfloat16).pin_memory()
    y = torch.zeros(256, 1, 64, dtype=torch.bfloat16).pin_memory()
    with pytest.raises(pt.PTError):
        hs.run(x, y, y, x, bm, x.clone(), y.clone(), y.clone())
    bm.free()
    hs.free()
