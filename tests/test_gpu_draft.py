"""Draft-block (DFlash) maps on the GPU against the oracle (oracle/draft.py):
block map and tile masks bit-exact, forward and backward within the bf16
(tensor-core) and fp32 (CUDA-core) tolerances, on layouts that span several
tiles with ragged tails, causal and bidirectional blocks, windows and
document-gated context."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import prefix_tree_block_gb300 as pt
from oracle import draft as OD
from prefix_tree_block_gb300 import workloads as W

from parity import FWD_ATOL, GRAD_RL2, LSE_ATOL, compare_blockmap, rel_l2

pytestmark = pytest.mark.gpu


def _layout(seed):
    """Seeded draft layout: context length, anchors, block size, keep flags,
    causal, window, documents."""
    rng = np.random.default_rng(seed)
    S = int(rng.integers(200, 700))
    bs = int(rng.choice([4, 8, 16, 24]))
    nb = int(rng.integers(4, 24))
    anchors = np.sort(rng.integers(1, S + 1, nb))
    keep = rng.random(nb) > 0.1
    causal = bool(seed % 2)
    window = int(rng.integers(32, 300)) if seed % 3 == 1 else 0
    if seed % 3 == 2:
        cuts = np.sort(rng.choice(np.arange(1, S), 3, replace=False))
        ctx_doc = np.searchsorted(cuts, np.arange(S), side="right").astype(np.int32)
        anchor_doc = ctx_doc[np.maximum(anchors - 1, 0)]
    else:
        ctx_doc = anchor_doc = None
    return dict(ctx_len=S, anchors=anchors, block_size=bs, block_keep=keep, causal=causal, window=window,
                ctx_doc=ctx_doc, anchor_doc=anchor_doc)


def _unpack(words):
    w = np.asarray(words, np.uint32)
    bits = (w[..., None] >> np.arange(32, dtype=np.uint32)) & 1
    return bits.reshape(w.shape[0], 128, 128).astype(bool)


@pytest.mark.parametrize("seed", range(6))
def test_draft_blockmap_and_masks_bit_exact(seed):
    lay = _layout(seed)
    mask = OD.draft_mask(**lay)
    bm = pt.build_blockmap_draft(**lay)
    got = bm.export()
    compare_blockmap(got, OD.mask_blockmap(mask, 128, 128))
    mk = bm.export_masks()
    T = mask.shape[0]
    pad = np.zeros((bm.nq * 128, bm.nk * 128), bool)
    pad[:T, :T] = mask.astype(bool)
    rows, cols = _unpack(mk["mask_rows"]), _unpack(mk["mask_cols"])
    for i in range(bm.nq):
        for e in range(got["q_ptr"][i], got["q_ptr"][i + 1]):
            j, s = got["kv_idx"][e], mk["pidx"][e]
            want = pad[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
            if got["kind"][e] == 1:
                assert s == -1 and want.all()
            else:
                np.testing.assert_array_equal(rows[s], want)
                np.testing.assert_array_equal(cols[s], want.T)
    bm.free()


@pytest.mark.parametrize("seed,D,dtype", [(0, 64, "bf16"), (1, 128, "bf16"), (2, 64, "bf16"), (4, 256, "bf16"),
                                          (3, 32, "f32"), (5, 64, "f32")])
def test_draft_attention_matches_oracle(seed, D, dtype):
    lay = _layout(seed)
    mask = OD.draft_mask(**lay)
    T = mask.shape[0]
    Hq, Hkv = 4, 2
    q, k, v, do = W.make_tensors(T, Hq, Hkv, D, dtype, 50 + seed)
    Q, K, V, dO = (x.cuda() for x in (q, k, v, do))
    bm = pt.build_blockmap_draft(**lay)
    O, L = pt.attn_fwd(Q, K, V, bm)
    dQ, dK, dV = pt.attn_bwd(dO, Q, K, V, O, L, bm)
    torch.cuda.synchronize()
    pt.sync_status()
    bm.free()
    Or, Lr = OD.masked_attn_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), mask)
    np.testing.assert_allclose(O.float().cpu().numpy(), Or, rtol=0, atol=FWD_ATOL[dtype])
    Lg = L.cpu().numpy()
    fin = np.isfinite(Lr)
    assert np.array_equal(np.isfinite(Lg), fin)
    np.testing.assert_allclose(Lg[fin], Lr[fin], rtol=0, atol=LSE_ATOL[dtype])
    gr = OD.masked_attn_bwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), do.double().numpy(), mask)
    for g, r in zip((dQ, dK, dV), gr):
        assert rel_l2(g.float().cpu().numpy(), r) <= GRAD_RL2[dtype]
    # context rows and dropped blocks: nothing kept, exact zeros
    empty = ~mask.astype(bool).any(axis=1)
    assert np.all(O.float().cpu().numpy()[empty] == 0)
    assert np.all(dQ.float().cpu().numpy()[empty] == 0)


def test_draft_dense_map_masks_every_tile():
    lay = _layout(2)
    mask = OD.draft_mask(**lay).astype(bool)
    bm = pt.build_blockmap_draft(**lay)
    d = bm.dense()
    lst, mk = d.export(), d.export_masks()
    T = mask.shape[0]
    pad = np.zeros((d.nq * 128, d.nk * 128), bool)
    pad[:T, :T] = mask
    rows = _unpack(mk["mask_rows"])
    for i in range(d.nq):
        for e in range(lst["q_ptr"][i], lst["q_ptr"][i + 1]):
            j, s = lst["kv_idx"][e], mk["pidx"][e]
            np.testing.assert_array_equal(rows[s], pad[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128])
    d.free()
    bm.free()


def test_draft_rejects_bad_arguments():
    with pytest.raises(pt.PTError):  # anchor past the context
        pt.build_blockmap_draft(10, [11], 4)
    with pytest.raises(pt.PTError):  # a document split into two runs
        pt.build_blockmap_draft(6, [3], 2, ctx_doc=[0, 0, 1, 1, 0, 0], anchor_doc=[0])
    with pytest.raises(pt.PTError):  # one of the two document arrays
        pt.build_blockmap_draft(6, [3], 2, ctx_doc=[0, 0, 0, 1, 1, 1])
    with pytest.raises(pt.PTError):  # tiles other than 128 x 128
        pt.build_blockmap_draft(64, [3], 2, block_m=64, block_n=64)
    with pytest.raises(pt.PTError):  # block size below 1
        pt.build_blockmap_draft(64, [3], 0)


@pytest.mark.parametrize("seed", [1, 2, 5])
def test_draft_tile_missing_from_host_lists_is_caught_on_device(seed):
    """Draft maps at 128 x 128 tiles are built from host lists too: the device
    classifies only the listed tiles and checks their kept pairs against the
    map's closed-form count, so a non-empty tile dropped from the host's lists
    (the test hook drops one) shows up as PT_ERR_INVALID_ARG at the next sync;
    the next build is clean and matches the oracle's map."""
    lib = pt.load_library()
    lay = _layout(seed)
    want = OD.mask_blockmap(OD.draft_mask(**lay), 128, 128)
    lib.pt_debug_drop_listed_tile(1)
    try:
        bm = pt.build_blockmap_draft(**lay)
        with pytest.raises(pt.PTError) as ei:
            pt.sync_status()
        assert ei.value.status == pt.PT_ERR_INVALID_ARG
        assert bm.nnz == want["nnz"] - 1
        bm.free()
    finally:
        lib.pt_debug_drop_listed_tile(0)
    bm = pt.build_blockmap_draft(**lay)
    pt.sync_status()
    compare_blockmap(bm.export(), want)
    bm.free()
