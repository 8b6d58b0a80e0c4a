"""Pins of the draft-block (DFlash) oracle (oracle/draft.py), on the CPU.

- The mask against hand-worked matrices (tests/golden/draft_mask_*.txt) and
  against a pair-by-pair transcription of the rule on random small layouts.
- The dense masked attention and tile classification against the tree
  oracle (oracle.c), itself pinned in test_oracle_pins.py, on tree masks.
- The backward against central finite differences of the forward.
"""
import os

import numpy as np
import pytest

from oracle import draft as OD
from oracle import oracle as OR

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    meta, rows = {}, []
    for line in open(os.path.join(GOLD, name)):
        line = line.strip()
        if line.startswith("#"):
            k, v = line[1:].split(":")
            meta[k.strip()] = [int(x) for x in v.split()]
        elif line:
            rows.append([int(x) for x in line.split()])
    return meta, np.array(rows, np.uint8)


def test_golden_bidirectional():
    meta, want = _read_golden("draft_mask_bidir.txt")
    got = OD.draft_mask(meta["ctx_len"][0], meta["anchors"], meta["block_size"][0], causal=bool(meta["causal"][0]),
                        window=meta["window"][0])
    np.testing.assert_array_equal(got, want)


def test_golden_causal_window_documents():
    meta, want = _read_golden("draft_mask_causal_window_docs.txt")
    got = OD.draft_mask(meta["ctx_len"][0], meta["anchors"], meta["block_size"][0], causal=bool(meta["causal"][0]),
                        window=meta["window"][0], ctx_doc=meta["ctx_doc"], anchor_doc=meta["anchor_doc"])
    np.testing.assert_array_equal(got, want)


def _pair_rule(S, anchors, bs, keep, causal, window, ctx_doc, anchor_doc, q, kv):
    # the rule, one (q, kv) pair at a time, in real positions
    if q < S:
        return 0  # context rows are not queries
    b, k = divmod(q - S, bs)
    if not keep[b]:
        return 0
    pos_q = anchors[b] + k
    if kv < S:
        if kv >= anchors[b]:
            return 0
        if ctx_doc is not None and ctx_doc[kv] != anchor_doc[b]:
            return 0
        if window > 0 and pos_q - kv >= window:
            return 0
        return 1
    b2, k2 = divmod(kv - S, bs)
    if b2 != b:
        return 0
    return 1 if (not causal or k2 <= k) else 0


@pytest.mark.parametrize("seed", range(6))
def test_mask_matches_pair_rule(seed):
    rng = np.random.default_rng(seed)
    S = int(rng.integers(1, 40))
    nb = int(rng.integers(1, 6))
    bs = int(rng.integers(1, 6))
    anchors = rng.integers(0, S + 1, nb)
    keep = rng.random(nb) > 0.2
    causal = bool(rng.integers(0, 2))
    window = int(rng.integers(0, 8)) if seed % 2 else 0
    if seed >= 3:
        cuts = np.sort(rng.integers(1, S + 1, 2))
        ctx_doc = np.searchsorted(cuts, np.arange(S), side="right")
        anchor_doc = rng.integers(0, 3, nb)
    else:
        ctx_doc = anchor_doc = None
    got = OD.draft_mask(S, anchors, bs, keep, causal, window, ctx_doc, anchor_doc)
    T = S + nb * bs
    want = np.array([[_pair_rule(S, anchors, bs, keep, causal, window, ctx_doc, anchor_doc, q, kv)
                      for kv in range(T)] for q in range(T)], np.uint8)
    np.testing.assert_array_equal(got, want)


def _random_tree(rng, n_nodes):
    lengths = rng.integers(0, 40, n_nodes)
    lengths[0] = max(lengths[0], 1)
    parent = [-1] + [int(rng.integers(0, i)) for i in range(1, n_nodes)]
    leaves = [i for i in range(n_nodes) if i not in parent[1:]]
    paths = []
    for leaf in leaves:
        p, n = [], leaf
        while n != -1:
            p.append(n)
            n = parent[n]
        paths.append(p[::-1])
    ptr = np.cumsum([0] + [len(p) for p in paths]).astype(np.int32)
    return lengths.astype(np.int32), ptr, np.concatenate(paths).astype(np.int32)


@pytest.mark.parametrize("seed", range(4))
def test_mask_blockmap_matches_tree_oracle(seed):
    rng = np.random.default_rng(100 + seed)
    nl, pp, pn = _random_tree(rng, 6)
    lab = OR.tree_labels(nl, pp, pn)
    mask = OR.dense_mask(lab)
    for BM, BN in ((16, 16), (32, 16), (8, 24)):
        got = OD.mask_blockmap(mask, BM, BN)
        want = OR.blockmap(lab, BM, BN)
        for key in ("q_ptr", "kv_idx", "kind", "k_ptr", "q_idx", "kindT"):
            np.testing.assert_array_equal(got[key], want[key], err_msg=f"{key} at {BM}x{BN}")


@pytest.mark.parametrize("seed", range(3))
def test_masked_attention_matches_tree_oracle(seed):
    rng = np.random.default_rng(200 + seed)
    nl, pp, pn = _random_tree(rng, 5)
    lab = OR.tree_labels(nl, pp, pn)
    T = lab.T
    Hq, Hkv, D = 4, 2, 8
    Q, K, V, dO = (rng.standard_normal((T, h, D)) for h in (Hq, Hkv, Hkv, Hq))
    mask = OR.dense_mask(lab)
    O, L = OD.masked_attn_fwd(Q, K, V, mask)
    O2, L2 = OR.attn_fwd(Q, K, V, lab)
    np.testing.assert_allclose(O, O2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, L2, rtol=0, atol=1e-12)
    got = OD.masked_attn_bwd(Q, K, V, dO, mask)
    want = OR.attn_bwd(Q, K, V, dO, lab)
    for g, w in zip(got, want):
        np.testing.assert_allclose(g, w, rtol=0, atol=1e-11)


def test_draft_rows_without_keys():
    # context rows and blocks with a false keep flag: O = 0, LSE = -inf, no gradient
    mask = OD.draft_mask(6, [3, 5], 2, block_keep=[True, False])
    rng = np.random.default_rng(7)
    Q, K, V, dO = (rng.standard_normal((10, 2, 4)) for _ in range(4))
    O, L = OD.masked_attn_fwd(Q, K, V, mask)
    assert np.all(O[:6] == 0) and np.all(np.isneginf(L[:, :6]))
    assert np.all(O[8:] == 0) and np.all(np.isneginf(L[:, 8:]))
    dQ, dK, dV = OD.masked_attn_bwd(Q, K, V, dO, mask)
    assert np.all(dQ[:6] == 0) and np.all(dQ[8:] == 0)
    assert np.all(dK[3:6] == 0) and np.all(dK[8:] == 0)  # keys nobody keeps


def test_draft_backward_finite_differences():
    rng = np.random.default_rng(11)
    mask = OD.draft_mask(7, [2, 6], 3, causal=False, window=4, ctx_doc=[0, 0, 0, 1, 1, 1, 1], anchor_doc=[0, 1])
    T = mask.shape[0]
    Q, K, V, dO = (rng.standard_normal((T, h, 3)) for h in (2, 1, 1, 2))
    dQ, dK, dV = OD.masked_attn_bwd(Q, K, V, dO, mask)

    def loss(Qx, Kx, Vx):
        return float((OD.masked_attn_fwd(Qx, Kx, Vx, mask)[0] * dO).sum())

    eps = 1e-6
    for X, G, which in ((Q, dQ, 0), (K, dK, 1), (V, dV, 2)):
        for idx in [(8, 1, 2), (1, 0, 0), (12, 0, 1), (9, 0, 2)]:
            if idx[1] >= X.shape[1]:
                idx = (idx[0], 0, idx[2])
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += eps
            Xm[idx] -= eps
            args_p = [Q, K, V]
            args_m = [Q, K, V]
            args_p[which], args_m[which] = Xp, Xm
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - G[idx]) <= 1e-6 * max(1.0, abs(fd)), (which, idx, fd, G[idx])
