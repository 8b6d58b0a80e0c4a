"""Draft-block (DFlash) attention mask and dense masked attention, fp64.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg may import this module; the library and its binding never do.

The mask follows the DFlash pages: "support sequence packing in the Domino and
JetSpec drafts" (a draft block's context prefix is restricted to its anchor's
document; the query side is the draft blocks only, the context is keys only)
and the DFlash-family drafter PR (the visibility rule: context before the
block, a window counted from each query's real position, block-causal when the
in-block attention is causal).  Readings where the pages are silent:

- Flat layout: the ctx_len context tokens first, then block b's block_size
  tokens at [ctx_len + b*bs, ctx_len + (b+1)*bs).  Block token k sits at real
  position anchor[b] + k.  Context rows are not queries: they keep nothing.
- Context key kv (0 <= kv < ctx_len) is kept by block b's token k iff
  kv < anchor[b] ("context before the block"), kv's document equals the
  anchor's document when document ids are given, and, with a window w > 0,
  (anchor[b] + k) - kv < w (the window counted from the query's real position;
  it applies to the context only).
- In-block key k' is kept by token k iff the in-block attention is
  bidirectional, or k' <= k when it is causal.  No block sees another block.
- A block whose keep flag is false keeps nothing (its rows return 0).

The attention functions are the plain definition over an explicit T x T keep
matrix (the same definition the tree oracle writes out per pair in oracle.c).
"""
from __future__ import annotations

from typing import Optional

import numpy as np


def draft_mask(ctx_len: int, anchors, block_size: int, block_keep=None, causal: bool = False, window: int = 0,
               ctx_doc=None, anchor_doc=None) -> np.ndarray:
    """The T x T keep matrix (uint8), T = ctx_len + len(anchors) * block_size."""
    anchors = np.asarray(anchors, dtype=np.int64)
    nb, bs, S = int(anchors.size), int(block_size), int(ctx_len)
    keep_b = np.ones(nb, bool) if block_keep is None else np.asarray(block_keep, dtype=bool)
    T = S + nb * bs
    m = np.zeros((T, T), np.uint8)
    kv = np.arange(S)
    for b in range(nb):
        if not keep_b[b]:
            continue
        a = int(anchors[b])
        ctx_ok = kv < a
        if ctx_doc is not None:
            ctx_ok &= np.asarray(ctx_doc)[:S] == np.asarray(anchor_doc)[b]
        r0 = S + b * bs
        for k in range(bs):
            row = ctx_ok.copy()
            if window > 0:
                row &= (a + k) - kv < window
            m[r0 + k, :S] = row
            m[r0 + k, r0:r0 + (k + 1 if causal else bs)] = 1
    return m


def mask_blockmap(mask: np.ndarray, BM: int, BN: int) -> dict:
    """Tile classes of a keep matrix: kind 0 (nothing kept), 1 (every in-range
    pair of a fully in-range tile kept), 2 (partial); q-major CSR and its
    kv-major transpose, as the tree oracle's blockmap returns them."""
    T = mask.shape[0]
    nq, nk = -(-T // BM), -(-T // BN)
    pad = np.zeros((nq * BM, nk * BN), np.int64)
    pad[:T, :T] = mask
    kept = pad.reshape(nq, BM, nk, BN).sum(axis=(1, 3))
    kind = np.where(kept == 0, 0, 2).astype(np.uint8)
    rows_in = np.minimum(BM, T - np.arange(nq) * BM)
    cols_in = np.minimum(BN, T - np.arange(nk) * BN)
    full = (kept == BM * BN) & (rows_in[:, None] == BM) & (cols_in[None, :] == BN)
    kind[full] = 1
    q_ptr, kv_idx, kinds = [0], [], []
    for i in range(nq):
        js = np.nonzero(kind[i])[0]
        kv_idx.extend(js.tolist())
        kinds.extend(kind[i, js].tolist())
        q_ptr.append(len(kv_idx))
    k_ptr, q_idx, kindT = [0], [], []
    for j in range(nk):
        is_ = np.nonzero(kind[:, j])[0]
        q_idx.extend(is_.tolist())
        kindT.extend(kind[is_, j].tolist())
        k_ptr.append(len(q_idx))
    return dict(q_ptr=np.array(q_ptr, np.int32), kv_idx=np.array(kv_idx, np.int32), kind=np.array(kinds, np.uint8),
                k_ptr=np.array(k_ptr, np.int32), q_idx=np.array(q_idx, np.int32), kindT=np.array(kindT, np.uint8),
                nnz=len(kv_idx), nq=nq, nk=nk)


def _scale(D: int, scale: float) -> float:
    return scale if scale > 0 else 1.0 / np.sqrt(D)


def masked_attn_fwd(Q, K, V, mask: np.ndarray, scale: float = 0.0):
    """O [T,Hq,D] and LSE [Hq,T] (natural log); rows keeping nothing give O = 0
    and LSE = -inf.  GQA: q head h reads kv head h // (Hq / Hkv)."""
    Q, K, V = (np.asarray(x, dtype=np.float64) for x in (Q, K, V))
    T, Hq, D = Q.shape
    g = Hq // K.shape[1]
    sc = _scale(D, scale)
    keep = mask.astype(bool)
    any_row = keep.any(axis=1)
    O = np.zeros((T, Hq, D))
    L = np.full((Hq, T), -np.inf)
    for h in range(Hq):
        s = sc * (Q[:, h, :] @ K[:, h // g, :].T)
        s = np.where(keep, s, -np.inf)
        m = np.where(any_row, s.max(axis=1), 0.0)
        e = np.where(keep, np.exp(s - m[:, None]), 0.0)
        l = e.sum(axis=1)
        ok = l > 0
        O[ok, h, :] = (e[ok] @ V[:, h // g, :]) / l[ok, None]
        L[h, ok] = m[ok] + np.log(l[ok])
    return O, L


def masked_attn_bwd(Q, K, V, dO, mask: np.ndarray, scale: float = 0.0):
    """dQ [T,Hq,D], dK and dV [T,Hkv,D] from the upstream gradient dO, with the
    forward recomputed here: P = exp(s - LSE), dV = sum_h P^T dO,
    dP = dO V^T, Delta = rowsum(dO * O), dS = P (dP - Delta), dQ = scale dS K,
    dK = scale sum_h dS^T Q."""
    Q, K, V, dO = (np.asarray(x, dtype=np.float64) for x in (Q, K, V, dO))
    T, Hq, D = Q.shape
    Hkv = K.shape[1]
    g = Hq // Hkv
    sc = _scale(D, scale)
    O, L = masked_attn_fwd(Q, K, V, mask, scale)
    keep = mask.astype(bool)
    dQ = np.zeros_like(Q)
    dK = np.zeros((T, Hkv, D))
    dV = np.zeros((T, Hkv, D))
    for h in range(Hq):
        hk = h // g
        s = sc * (Q[:, h, :] @ K[:, hk, :].T)
        lse = np.where(np.isfinite(L[h]), L[h], np.inf)
        P = np.where(keep, np.exp(s - lse[:, None]), 0.0)
        dV[:, hk, :] += P.T @ dO[:, h, :]
        dP = dO[:, h, :] @ V[:, hk, :].T
        delta = (dO[:, h, :] * O[:, h, :]).sum(axis=1)
        dS = P * (dP - delta[:, None])
        dQ[:, h, :] = sc * (dS @ K[:, hk, :])
        dK[:, hk, :] += sc * (dS.T @ Q[:, h, :])
    return dQ, dK, dV
