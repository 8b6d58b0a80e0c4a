"""Pins of the shared-prefix fold oracle (oracle/fold.py), on the CPU.

- Hand-worked folds of small rollout batches (tests/golden/fold_*.txt):
  flat sequence, position ids, unfolded rows and the summed gradient.
- The shared-prefix group in closed form: [prompt | c_0 | c_1 | ...] built
  with torch.cat from the group sizes alone, position ids P.., and torch
  autograd of that construction for the gradient of the unfold.
- The adjoint identity <unfold(Y), Z> = <Y, unfold_grad(Z)> and the round
  trip fold(unfold(Y)) = Y on random trees.
- The point of the fold ("cp=1 shared-prefix prefix-tree attention for
  rollouts", PR description): prefix-tree attention over the folded
  sequence, unfolded, equals plain causal attention over every rollout row.
- Planted disagreements between rollouts are counted; malformed input raises.
"""
import os

import numpy as np
import pytest
import torch

from oracle import fold as OF
from oracle import oracle as OR
from prefix_tree_block_gb300 import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")
FIXTURES = ["fold_grpo_P3.txt", "fold_two_groups.txt", "fold_tree_depth3.txt"]


def _read(name):
    d = {"roll": [], "droll": []}
    for line in open(os.path.join(GOLD, name)):
        line = line.split("#")[0].strip()
        if not line:
            continue
        key, rest = line.split(None, 1)
        if key == "paths":
            d["paths"] = [[int(x) for x in p.split()] for p in rest.split("|")]
        elif key in ("roll", "droll"):
            d[key].append([int(x) for x in rest.split()])
        else:
            d[key] = [int(x) for x in rest.split()]
    st = W.tree_structure(d["node_lengths"], d["paths"])
    return st, d


@pytest.mark.parametrize("name", FIXTURES)
def test_golden(name):
    st, d = _read(name)
    tree = (st.node_lengths, st.path_ptr, st.path_nodes)
    L = d["row_len"][0]
    roll = np.array(d["roll"], np.int64)
    np.testing.assert_array_equal(OF.fold(roll, *tree), d["flat"])
    np.testing.assert_array_equal(OF.positions(*tree), d["positions"])
    np.testing.assert_array_equal(OF.unfold(np.array(d["flat"], np.int64), *tree, L), roll)
    np.testing.assert_array_equal(OF.unfold_grad(np.array(d["droll"], np.float64), *tree), d["dflat"])
    assert OF.mismatches(roll, *tree) == 0
    assert OF.max_row_length(*tree) <= L


def test_planted_disagreements_are_counted():
    st, d = _read("fold_grpo_P3.txt")
    tree = (st.node_lengths, st.path_ptr, st.path_nodes)
    roll = np.array(d["roll"], np.int64)
    bad = roll.copy()
    bad[1, 0] = 99  # a later sample's copy of a prompt token
    assert OF.mismatches(bad, *tree) == 1
    bad = roll.copy()
    bad[0, 2] = 99  # the first sample's prompt token: every other copy now disagrees
    assert OF.mismatches(bad, *tree) == 2
    assert OF.fold(bad, *tree)[2] == 99  # the fold keeps the first sample's value
    bad = roll.copy()
    bad[0, 5] = 99  # padding is not compared
    bad[1, 3] = 98  # a completion token exists once and cannot disagree
    assert OF.mismatches(bad, *tree) == 0


def _grpo_specs(rng, n_groups):
    specs = []
    for g in range(n_groups):
        P = int(rng.integers(0, 9)) if g else 0
        specs.append((P, [int(rng.integers(0, 7)) for _ in range(int(rng.integers(1, 5)))]))
    return specs


@pytest.mark.parametrize("seed", range(4))
def test_grpo_closed_form_and_autograd(seed):
    rng = np.random.default_rng(seed)
    specs = _grpo_specs(rng, 3)
    st = W.grpo_structure(specs)
    tree = (st.node_lengths, st.path_ptr, st.path_nodes)
    L = max(P + r for P, Rs in specs for r in Rs) + 2
    C = 3
    flat = torch.randn(st.T, C, dtype=torch.float64, requires_grad=True)
    # [prompt | c_0 | c_1 | ...] per group, rows = prompt ++ own completion, padded with zeros
    rows, pos, base = [], [], 0
    for P, Rs in specs:
        pr = flat[base:base + P]
        c0 = base + P
        for r in Rs:
            row = torch.cat([pr, flat[c0:c0 + r], torch.zeros(L - P - r, C, dtype=torch.float64)])
            rows.append(row)
            c0 += r
        pos += list(range(P)) + [P + k for r in Rs for k in range(r)]
        base = c0
    roll = torch.stack(rows)
    np.testing.assert_array_equal(OF.positions(*tree), pos)
    np.testing.assert_array_equal(OF.unfold(flat.detach().numpy(), *tree, L), roll.detach().numpy())
    np.testing.assert_array_equal(OF.fold(roll.detach().numpy(), *tree), flat.detach().numpy())
    Z = torch.randn(roll.shape, dtype=torch.float64)
    (roll * Z).sum().backward()
    np.testing.assert_allclose(OF.unfold_grad(Z.numpy(), *tree), flat.grad.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", range(6))
def test_adjoint_and_round_trip_on_random_trees(seed):
    rng = np.random.default_rng(100 + seed)
    st = W.random_tree(rng, int(rng.integers(2, 12)), 6)
    tree = (st.node_lengths, st.path_ptr, st.path_nodes)
    L = OF.max_row_length(*tree) + int(rng.integers(0, 3))
    Y = rng.standard_normal((st.T, 4))
    Z = rng.standard_normal((st.n_samples, L, 4))
    U = OF.unfold(Y, *tree, L)
    lhs = float((U * Z).sum())
    rhs = float((Y * OF.unfold_grad(Z, *tree)).sum())
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))
    np.testing.assert_array_equal(OF.fold(U, *tree), Y)
    assert OF.mismatches(U, *tree) == 0
    # every flat token appears in the rollouts as many times as paths run through its node
    counts = OF.unfold_grad(np.ones((st.n_samples, L)), *tree)
    node_of = np.repeat(np.arange(st.n_nodes), st.node_lengths)
    through = np.array([sum(n in p for p in st.paths()) for n in range(st.n_nodes)])
    np.testing.assert_array_equal(counts, through[node_of])


def _causal_attention(q, k, v, scale):
    # textbook causal softmax attention of one sequence; q [n,Hq,D], k/v [n,Hkv,D]
    n, Hq, D = q.shape
    g = Hq // k.shape[1]
    out = np.zeros_like(q)
    for h in range(Hq):
        s = scale * q[:, h] @ k[:, h // g].T
        s[np.triu_indices(n, 1)] = -np.inf
        p = np.exp(s - s.max(axis=1, keepdims=True))
        out[:, h] = (p / p.sum(axis=1, keepdims=True)) @ v[:, h // g]
    return out


@pytest.mark.parametrize("kind", ["grpo", "tree"])
def test_folded_attention_equals_per_rollout_causal_attention(kind):
    rng = np.random.default_rng(7)
    if kind == "grpo":
        st = W.grpo_structure([(5, [3, 1, 4]), (0, [2, 6]), (4, [0, 2])])
    else:
        st = W.random_tree(rng, 9, 5)
    tree = (st.node_lengths, st.path_ptr, st.path_nodes)
    Hq, Hkv, D = 4, 2, 8
    q, k, v = (rng.standard_normal((st.T, h, D)) for h in (Hq, Hkv, Hkv))
    O, _ = OR.attn_fwd(q, k, v, OR.structure_labels(st))
    L = OF.max_row_length(*tree)
    Ou = OF.unfold(O, *tree, L)
    qu, ku, vu = (OF.unfold(x, *tree, L) for x in (q, k, v))
    for s, row in enumerate(OF.sample_rows(*tree)):
        n = row.size
        if n == 0:
            continue
        want = _causal_attention(qu[s, :n], ku[s, :n], vu[s, :n], 1.0 / np.sqrt(D))
        np.testing.assert_allclose(Ou[s, :n], want, rtol=0, atol=1e-12)


def test_malformed_input_raises():
    st = W.grpo_structure([(3, [2, 1])])
    tree = (st.node_lengths, st.path_ptr, st.path_nodes)
    with pytest.raises(OF.FoldError):
        OF.unfold(np.zeros(st.T), *tree, 4)  # a row of 5 tokens does not fit in 4
    orphan = W.tree_structure([2, 1, 1], [[0, 1]])  # node 2 is on no path
    with pytest.raises(OF.FoldError):
        OF.positions(orphan.node_lengths, orphan.path_ptr, orphan.path_nodes)
    twisted = W.tree_structure([1, 1, 1], [[0, 1, 2], [0, 2]])  # node 2 at two depths
    with pytest.raises(OF.FoldError):
        OF.positions(twisted.node_lengths, twisted.path_ptr, twisted.path_nodes)
