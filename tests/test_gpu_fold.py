"""Parity of the shared-prefix fold kernels (pt_fold_plan, pt_fold, pt_unfold,
pt_unfold_grad, pt_fold_positions, pt_fold_mismatches) with the oracle
(oracle/fold.py), through the C ABI.

Byte and index work (fold, unfold, positions, mismatch counts) must match
bit for bit.  The gradient sums run in fp32 in sample order and are rounded
once, so against the exact fp64 sum of n copies they may differ by the fp32
accumulation, at most n * 2^-24 * sum|x| (plus the same again for rounding
the inputs' partial sums), and for bf16 by the final rounding, half an ulp:
2^-9 * |exact|; the tests allow 2^-8 relative plus 2 * n * 2^-24 * sum|x|.
"""
import numpy as np
import pytest
import torch

import prefix_tree_block_gb300 as pt
from oracle import fold as OF
from oracle import oracle as OR
from prefix_tree_block_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _tree(st):
    return st.node_lengths, st.path_ptr, st.path_nodes


def _structures():
    rng = np.random.default_rng(11)
    yield "grpo", W.grpo_structure([(5, [3, 1, 4]), (0, [2, 6]), (4, [0, 2]), (7, [])]), 0
    yield "one_completion", W.grpo_structure([(9, [4])]), 3
    yield "empty_prompts", W.grpo_structure([(0, [1, 1, 5])]), 1
    for i in range(3):
        yield f"random_tree{i}", W.random_tree(rng, int(rng.integers(3, 14)), 40), int(rng.integers(0, 5))
    yield "ragged_wide", W.grpo_structure([(131, [29, 100, 1, 64]), (1, [250, 3])]), 7
    yield "twelve_samples", W.grpo_structure([(37, [5, 9, 1, 3, 12, 7, 2, 8, 4, 6, 10, 11])]), 2  # > 8 copies


STRUCTS = list(_structures())


def _rollouts(st, L, trailing, dtype, seed):
    """Consistent rollouts: the unfold (oracle) of random flat rows."""
    g = torch.Generator().manual_seed(seed)
    if dtype in (torch.int32, torch.int64, torch.uint8):
        flat = torch.randint(0, 120, (st.T,) + trailing, generator=g).to(dtype)
    else:
        flat = torch.randn((st.T,) + trailing, generator=g).to(dtype)
    roll = torch.from_numpy(OF.unfold(flat.numpy() if dtype != torch.bfloat16 else flat.view(torch.int16).numpy(),
                                      *_tree(st), L))
    if dtype == torch.bfloat16:
        roll = roll.view(torch.bfloat16)
    return flat, roll


@pytest.mark.parametrize("name,st,extra", STRUCTS, ids=[s[0] for s in STRUCTS])
@pytest.mark.parametrize("dtype,trailing", [(torch.int32, ()), (torch.int64, ()), (torch.uint8, (3,)),
                                            (torch.bfloat16, (96,)), (torch.float32, (5,))],
                         ids=["ids32", "ids64", "bytes3", "bf16x96", "f32x5"])
def test_fold_unfold_positions_bit_exact(name, st, extra, dtype, trailing):
    L = OF.max_row_length(*_tree(st)) + extra
    flat, roll = _rollouts(st, L, trailing, dtype, seed=len(name) + st.T)
    plan = pt.fold_plan(*_tree(st), L)
    assert (plan.T, plan.n_samples, plan.row_len) == (st.T, st.n_samples, L)
    got = plan.fold(roll.cuda()).cpu()
    assert torch.equal(got, flat)
    back = plan.unfold(flat.cuda()).cpu()
    assert torch.equal(back, roll)
    pos = plan.positions().cpu().numpy()
    np.testing.assert_array_equal(pos, OF.positions(*_tree(st)))
    assert plan.mismatches(roll.cuda()) == 0
    pt.sync_status()


def _grad_tolerance_ok(got, droll64, st, want, bf16):
    # |got - exact| <= 2^-8 |exact| (bf16 only) + 2 n 2^-24 sum|x| over the copies of each token
    absd = np.abs(droll64)
    summ = OF.unfold_grad(absd, *_tree(st))
    copies = OF.unfold_grad(np.ones(droll64.shape[:2]), *_tree(st))
    n = copies.reshape((-1,) + (1,) * (want.ndim - 1))
    bound = 2 * n * 2.0 ** -24 * summ + (2.0 ** -8 * np.abs(want) if bf16 else 0.0) + 1e-30
    err = np.abs(got - want)
    return bool((err <= bound).all()), float((err / bound).max())


@pytest.mark.parametrize("name,st,extra", STRUCTS, ids=[s[0] for s in STRUCTS])
@pytest.mark.parametrize("dtype,width", [(torch.float32, 64), (torch.float32, 7), (torch.bfloat16, 128),
                                         (torch.bfloat16, 3)], ids=["f32x64", "f32x7", "bf16x128", "bf16x3"])
def test_unfold_grad(name, st, extra, dtype, width):
    L = OF.max_row_length(*_tree(st)) + extra
    g = torch.Generator().manual_seed(st.T + width)
    droll = torch.randn(st.n_samples, L, width, generator=g).to(dtype)
    got = pt.fold_plan(*_tree(st), L).unfold_grad(droll.cuda()).cpu().double().numpy()
    d64 = droll.double().numpy()
    want = OF.unfold_grad(d64, *_tree(st))
    ok, worst = _grad_tolerance_ok(got, d64, st, want, dtype == torch.bfloat16)
    assert ok, f"worst error / bound = {worst}"
    # the padding entries are ignored: poisoning them changes nothing
    pad = torch.from_numpy(OF.unfold(np.ones((st.T, 1)), *_tree(st), L)[..., 0] == 0)
    droll[pad] = float("nan")
    got2 = pt.fold_plan(*_tree(st), L).unfold_grad(droll.cuda()).cpu().double().numpy()
    np.testing.assert_array_equal(got2, got)


def test_mismatches_counts_planted_differences():
    st = W.grpo_structure([(6, [2, 3, 1]), (4, [5, 2])])
    L = 12
    flat, roll = _rollouts(st, L, (8,), torch.int32, seed=3)
    plan = pt.fold_plan(*_tree(st), L)
    bad = roll.clone()
    bad[1, 2, 5] += 1  # a later sample's copy of a prompt token
    bad[0, 0, 0] += 1  # the first sample's prompt token: the other two copies now differ
    bad[3, 9, 1] += 1  # padding: not compared
    want = OF.mismatches(bad.numpy(), *_tree(st))
    assert want == 3
    assert plan.mismatches(bad.cuda()) == want


def test_workload_rollouts_full_size():
    """The GRPO-batch workload (8 groups, P=512, 8 completions of U[64,256])
    as rollout rows of hidden states (14 heads x 64 = 896 bf16 per token)."""
    st = W.config_structure(2)
    L = OF.max_row_length(*_tree(st))
    flat, roll = _rollouts(st, L, (896,), torch.bfloat16, seed=2)
    plan = pt.fold_plan(*_tree(st), L)
    rc = roll.cuda()
    assert torch.equal(plan.fold(rc).cpu(), flat)
    assert torch.equal(plan.unfold(flat.cuda()).cpu(), roll)
    assert plan.mismatches(rc) == 0
    np.testing.assert_array_equal(plan.positions().cpu().numpy(), OF.positions(*_tree(st)))
    # the gradient of the flat rows for a gradient on every rollout entry
    g = torch.Generator().manual_seed(5)
    droll = torch.randn(st.n_samples, L, 896, generator=g).to(torch.bfloat16)
    got = plan.unfold_grad(droll.cuda()).cpu().double().numpy()
    d64 = droll.double().numpy()
    want = OF.unfold_grad(d64, *_tree(st))
    ok, worst = _grad_tolerance_ok(got, d64, st, want, True)
    assert ok, f"worst error / bound = {worst}"


def test_folded_attention_unfolds_to_per_rollout_attention():
    """Fold rollout Q/K/V, run the prefix-tree forward on the flat layout,
    unfold O: equal (bf16 tolerance) to the oracle's attention unfolded."""
    st = W.grpo_structure([(200, [90, 150, 37]), (0, [64, 129])])
    Hq, Hkv, D = 4, 2, 128
    q, k, v, _ = W.make_tensors(st.T, Hq, Hkv, D, "bf16", seed=9)
    L = OF.max_row_length(*_tree(st))
    plan = pt.fold_plan(*_tree(st), L)
    rq, rk, rv = (plan.unfold(x.cuda()) for x in (q, k, v))  # rollout rows, as a trainer would hold them
    Q, K, V = (plan.fold(x) for x in (rq, rk, rv))
    bm = pt.build_blockmap_tree(*_tree(st), 128, 128)
    O, _ = pt.attn_fwd(Q, K, V, bm)
    Ou = plan.unfold(O).float().cpu().numpy()
    Ow, _ = OR.attn_fwd(q, k, v, OR.structure_labels(st))
    want = OF.unfold(Ow, *_tree(st), L)
    assert np.abs(Ou - want).max() <= 2e-2


def test_invalid_plans_rejected():
    st = W.grpo_structure([(3, [2, 1])])
    with pytest.raises(pt.PTError):
        pt.fold_plan(*_tree(st), 4)  # a 5-token row does not fit in 4
    with pytest.raises(pt.PTError):
        pt.fold_plan([2, 1, 1], [0, 2], [0, 1], 8)  # node 2 on no path


def test_empty_and_padding_only_rows():
    """No tokens at all, and a sample whose path holds only zero-length nodes (its row is all padding)."""
    empty = W.grpo_structure([(0, [0, 0])])
    plan = pt.fold_plan(*_tree(empty), 3)
    assert plan.T == 0
    roll = torch.full((2, 3, 4), 7, dtype=torch.int32, device="cuda")
    assert plan.fold(roll).numel() == 0
    assert torch.equal(plan.unfold(torch.empty(0, 4, dtype=torch.int32, device="cuda")).cpu(),
                       torch.zeros(2, 3, 4, dtype=torch.int32))
    assert plan.unfold_grad(torch.randn(2, 3, 8, device="cuda")).numel() == 0
    assert plan.positions().numel() == 0 and plan.mismatches(roll) == 0
    st = W.tree_structure([0, 0, 5, 3], [[0, 1], [0, 2, 3]])  # sample 0: zero-length nodes only
    L = 9
    flat, roll = _rollouts(st, L, (16,), torch.bfloat16, seed=4)
    plan = pt.fold_plan(*_tree(st), L)
    assert torch.equal(plan.fold(roll.cuda()).cpu(), flat)
    assert torch.equal(plan.unfold(flat.cuda()).cpu(), roll)
    droll = torch.randn(st.n_samples, L, 16).to(torch.bfloat16)
    got = plan.unfold_grad(droll.cuda()).cpu().double().numpy()
    want = OF.unfold_grad(droll.double().numpy(), *_tree(st))
    np.testing.assert_allclose(got, want, rtol=2.0 ** -8, atol=0)
