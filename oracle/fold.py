"""Shared-prefix fold and unfold of rollouts, by their definition (numpy).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg may import this module; the library and its binding never do.

The fold follows "cp=1 shared-prefix prefix-tree attention for rollouts"
(PR description): a group of one prompt and N sampled completions is stored
once as the flat sequence [prompt | c_0 | c_1 | ...], each completion's
position ids continue from its prompt, and the tree is handed on as
(node_lengths, sample_paths).  Written for the general tree, of which the
shared-prefix group is the depth-2 case:

- Flat layout: node i owns tokens [off_i, off_i + node_lengths[i]), off the
  exclusive prefix sum in id order (the layout the attention works on).
- Rollout layout: sample s is one row of length L (the row stride); its
  tokens are those of its path's nodes, root first, at positions 0, 1, ...;
  positions past the path's length are padding.
- fold (rollouts -> flat): a token shared by several samples is taken from
  the first sample (lowest index) whose path holds it; the others are
  expected to carry the same value (the fold is a deduplication).
- position id of a flat token: its position in any sample row that holds it
  (the same in all of them: a node's ancestors are the same whichever path
  reaches it).
- unfold (flat -> rollouts): every sample row gets its tokens back; shared
  tokens are copied into every row that holds them; padding is zero.
- unfold_grad: the adjoint of unfold, the gradient of a loss on the rollout
  rows with respect to the flat rows: a flat token receives the sum of the
  gradients of all its copies (exact fp64 sum here).
- mismatches: the number of (sample, position) entries whose value differs
  from the value the fold keeps for that token (0 when the rollouts really
  share their prefixes).
"""
from __future__ import annotations

from typing import List, Sequence

import numpy as np


class FoldError(ValueError):
    pass


def _paths(path_ptr, path_nodes) -> List[List[int]]:
    ptr = np.asarray(path_ptr, dtype=np.int64)
    nodes = np.asarray(path_nodes, dtype=np.int64)
    return [[int(x) for x in nodes[ptr[s]:ptr[s + 1]]] for s in range(ptr.size - 1)]


def sample_rows(node_lengths, path_ptr, path_nodes) -> List[np.ndarray]:
    """Flat token indices of every sample row, in row order: the tokens of the
    path's nodes, root first."""
    lengths = np.asarray(node_lengths, dtype=np.int64)
    off = np.concatenate([[0], np.cumsum(lengths)])
    rows = []
    for p in _paths(path_ptr, path_nodes):
        if not p:
            raise FoldError("empty sample path")
        for n in p:
            if not 0 <= n < lengths.size:
                raise FoldError(f"node {n} out of range")
        rows.append(np.concatenate([np.arange(off[n], off[n] + lengths[n]) for n in p]).astype(np.int64))
    return rows


def token_source(node_lengths, path_ptr, path_nodes):
    """For every flat token: (sample, position) of its first occurrence, and
    its position id.  Raises when a token is on no path or sits at two
    different positions (an inconsistent tree)."""
    lengths = np.asarray(node_lengths, dtype=np.int64)
    T = int(lengths.sum())
    src_s = np.full(T, -1, np.int64)
    pos = np.full(T, -1, np.int64)
    for s, row in enumerate(sample_rows(node_lengths, path_ptr, path_nodes)):
        for j, t in enumerate(row):
            if src_s[t] < 0:
                src_s[t], pos[t] = s, j
            elif pos[t] != j:
                raise FoldError(f"token {t} sits at positions {pos[t]} and {j}")
    if T and (src_s < 0).any():
        raise FoldError(f"token {int(np.argmax(src_s < 0))} is on no sample path")
    return src_s, pos


def positions(node_lengths, path_ptr, path_nodes) -> np.ndarray:
    """Position id of every flat token (int64 [T])."""
    return token_source(node_lengths, path_ptr, path_nodes)[1]


def _check_rows(roll, rows, L):
    if roll.shape[0] != len(rows) or roll.shape[1] != L:
        raise FoldError(f"rollouts have shape {roll.shape[:2]}, want ({len(rows)}, {L})")
    for s, r in enumerate(rows):
        if r.size > L:
            raise FoldError(f"sample {s} has {r.size} tokens, longer than the row length {L}")


def fold(roll: np.ndarray, node_lengths, path_ptr, path_nodes) -> np.ndarray:
    """roll [S, L, ...] -> flat [T, ...]: each token from its first sample."""
    roll = np.asarray(roll)
    rows = sample_rows(node_lengths, path_ptr, path_nodes)
    _check_rows(roll, rows, roll.shape[1])
    src_s, pos = token_source(node_lengths, path_ptr, path_nodes)
    out = np.zeros((src_s.size,) + roll.shape[2:], roll.dtype)
    for t in range(src_s.size):
        out[t] = roll[src_s[t], pos[t]]
    return out


def unfold(flat: np.ndarray, node_lengths, path_ptr, path_nodes, L: int) -> np.ndarray:
    """flat [T, ...] -> roll [S, L, ...]: every row gets its tokens, padding 0."""
    flat = np.asarray(flat)
    rows = sample_rows(node_lengths, path_ptr, path_nodes)
    out = np.zeros((len(rows), L) + flat.shape[1:], flat.dtype)
    _check_rows(out, rows, L)
    for s, r in enumerate(rows):
        for j, t in enumerate(r):
            out[s, j] = flat[t]
    return out


def unfold_grad(droll: np.ndarray, node_lengths, path_ptr, path_nodes) -> np.ndarray:
    """droll [S, L, ...] -> dflat [T, ...] (fp64): the sum over every copy of
    a token; padding entries of droll are ignored."""
    droll = np.asarray(droll, dtype=np.float64)
    rows = sample_rows(node_lengths, path_ptr, path_nodes)
    _check_rows(droll, rows, droll.shape[1])
    T = int(np.asarray(node_lengths, dtype=np.int64).sum())
    out = np.zeros((T,) + droll.shape[2:], np.float64)
    for s, r in enumerate(rows):
        for j, t in enumerate(r):
            out[t] += droll[s, j]
    return out


def mismatches(roll: np.ndarray, node_lengths, path_ptr, path_nodes) -> int:
    """How many (sample, position) entries differ from the value the fold
    keeps for their token (entries compared whole, byte for byte)."""
    roll = np.ascontiguousarray(roll)
    rows = sample_rows(node_lengths, path_ptr, path_nodes)
    _check_rows(roll, rows, roll.shape[1])
    src_s, pos = token_source(node_lengths, path_ptr, path_nodes)
    raw = roll.reshape(roll.shape[0], roll.shape[1], -1).view(np.uint8)
    n = 0
    for s, r in enumerate(rows):
        for j, t in enumerate(r):
            n += int(not np.array_equal(raw[s, j], raw[src_s[t], pos[t]]))
    return n


def max_row_length(node_lengths, path_ptr, path_nodes) -> int:
    return max((r.size for r in sample_rows(node_lengths, path_ptr, path_nodes)), default=0)
