"""Parity at the measured sizes: every element of O, LSE, dQ, dK and dV
against the fp64 oracle, on the workloads the benchmark times, in the launch
configuration it times (a 128 x 128 map built from the host tree arrays, the
forward, the backward with a full-size workspace so that long kv-major
columns are split across SMs).

- Workloads 2, 4 and 5 run whole (all heads, all rows and columns).
- Workload 3 (the long-prompt shape) and workload 6 (draft blocks) run whole
  on the GPU; every output element of their last kv head (its q heads' O,
  LSE and dQ, its dK and dV) is compared with the oracle run on that kv
  head's slice of the inputs, a problem of its own with Hq = Hq/Hkv, Hkv = 1
  on the same layout (the heads do not interact).

Tolerances are the parity tolerances of every other test: forward max-abs
2e-2 (LSE 2e-3), gradients relative L2 norm 3e-2 (bf16)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import prefix_tree_block_gb300 as pt
from oracle import draft as OD
from oracle import oracle as orc
from prefix_tree_block_gb300 import workloads as W
from parity import FWD_ATOL, GRAD_RL2, LSE_ATOL, ensure_built, rel_l2, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _run(bm, q, k, v, do):
    Q, K, V, dO = (to_dev(x) for x in (q, k, v, do))
    O, L = pt.attn_fwd(Q, K, V, bm)
    dQ, dK, dV = pt.attn_bwd(dO, Q, K, V, O, L, bm)
    pt.sync_status()
    return [x.float().cpu().numpy() for x in (O, L, dQ, dK, dV)]


def _compare(got, fwd, bwd):
    O, L, dQ, dK, dV = got
    Ow, Lw = fwd
    assert np.isfinite(O).all() and np.isfinite(dQ).all() and np.isfinite(dK).all() and np.isfinite(dV).all()
    err = np.abs(O - Ow).max()
    assert err <= FWD_ATOL["bf16"], f"O max-abs {err}"
    fin = np.isfinite(Lw)
    assert np.array_equal(np.isfinite(L), fin)
    lerr = np.abs(L[fin] - Lw[fin]).max() if fin.any() else 0.0
    assert lerr <= LSE_ATOL["bf16"], f"LSE max-abs {lerr}"
    errs = [rel_l2(g, w) for g, w in zip((dQ, dK, dV), bwd)]
    assert max(errs) <= GRAD_RL2["bf16"], errs


def _slice(x, a, b):
    return x[:, a:b].contiguous()


def _check_case(bm, q, k, v, do, oracle, slice_kv=None):
    """Run the whole problem on the GPU; compare with oracle(q, k, v, do) ->
    ((O, LSE), (dQ, dK, dV)) on all heads, or on kv head slice_kv and its q
    heads only."""
    got = _run(bm, q, k, v, do)
    bm.free()
    if slice_kv is not None:
        g = q.shape[1] // k.shape[1]
        a, b = slice_kv * g, (slice_kv + 1) * g
        q, do = _slice(q, a, b), _slice(do, a, b)
        k, v = _slice(k, slice_kv, slice_kv + 1), _slice(v, slice_kv, slice_kv + 1)
        O, L, dQ, dK, dV = got
        got = [O[:, a:b], L[a:b], dQ[:, a:b], dK[:, slice_kv:slice_kv + 1], dV[:, slice_kv:slice_kv + 1]]
    fwd, bwd = oracle(q, k, v, do)
    _compare(got, fwd, bwd)
    return got


def _tree_oracle(st):
    lab = orc.structure_labels(st)
    return lambda q, k, v, do: (orc.attn_fwd(q, k, v, lab), orc.attn_bwd(q, k, v, do, lab))


def _tree_map(st):
    return pt.build_blockmap_tree(st.node_lengths, st.path_ptr, st.path_nodes, 128, 128)


@pytest.mark.parametrize("c", [2, 4, 5])
def test_workload_every_element(c):
    cfg = W.CONFIGS[c]
    st = W.config_structure(c)
    q, k, v, do = W.make_tensors(st.T, cfg["Hq"], cfg["Hkv"], cfg["D"], "bf16", seed=c)
    _check_case(_tree_map(st), q, k, v, do, _tree_oracle(st))


def test_long_prompt_last_kv_head_every_element():
    cfg = W.CONFIGS[3]
    st = W.config_structure(3)
    q, k, v, do = W.make_tensors(st.T, cfg["Hq"], cfg["Hkv"], cfg["D"], "bf16", seed=3)
    _check_case(_tree_map(st), q, k, v, do, _tree_oracle(st), slice_kv=cfg["Hkv"] - 1)


def test_draft_workload_last_kv_head_every_element():
    cfg = W.CONFIGS[6]
    st = W.config_structure(6)
    kw = st.kwargs()
    q, k, v, do = W.make_tensors(st.T, cfg["Hq"], cfg["Hkv"], cfg["D"], "bf16", seed=6)
    mask = OD.draft_mask(**kw)

    def oracle(q, k, v, do):
        qd, kd, vd, dod = (x.double().numpy() for x in (q, k, v, do))
        return OD.masked_attn_fwd(qd, kd, vd, mask), OD.masked_attn_bwd(qd, kd, vd, dod, mask)

    got = _check_case(pt.build_blockmap_draft(**kw), q, k, v, do, oracle, slice_kv=cfg["Hkv"] - 1)
    # context rows keep nothing: exact zeros
    empty = ~mask.astype(bool).any(axis=1)
    assert np.all(got[0][empty] == 0) and np.all(got[2][empty] == 0)


def test_head_dim_512_every_element():
    """Workload 7 (packed documents at head_dim 512, the measurement shape of
    the tensor-core kernels at that head dim): every element of O, LSE, dQ,
    dK and dV."""
    cfg = W.CONFIGS[7]
    st = W.config_structure(7)
    q, k, v, do = W.make_tensors(st.T, cfg["Hq"], cfg["Hkv"], cfg["D"], "bf16", seed=7)
    _check_case(_tree_map(st), q, k, v, do, _tree_oracle(st))
