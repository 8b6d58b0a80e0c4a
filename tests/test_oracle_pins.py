"""Pins for the fp64 oracle: each test checks it against something other than
itself -- hand-written masks, an independent transcription of the segment
mask rule, textbook causal attention on the unfolded sequences, library
routines (torch SDPA and autograd in fp64), closed forms, invariants and
finite differences.  CPU only."""
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import oracle as orc
from prefix_tree_block_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# helpers written independently of the oracle
# ---------------------------------------------------------------------------

def p2_mask_mod(group_id, suffix_id):
    """Literal transcription of the segment-form keep rule of
    "prefix_grouper_kernel.py" (_make_mask_mod):
        same_group & ((is_prefix[kv] & kv <= q) | (same_suffix & ~is_prefix[q] & kv <= q))."""
    g = np.asarray(group_id)
    s = np.asarray(suffix_id)
    T = g.size
    q = np.arange(T)[:, None]
    kv = np.arange(T)[None, :]
    is_prefix = s == -1
    same_group = g[:, None] == g[None, :]
    causal = kv <= q
    same_suffix = (s[None, :] == s[:, None]) & (~is_prefix[:, None])
    return (same_group & ((is_prefix[None, :] & causal) | (same_suffix & causal))).astype(np.uint8)


def read_golden_mask(name):
    rows, meta = [], {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line.startswith("#"):
                k, _, v = line[1:].partition(":")
                meta[k.strip()] = v.strip()
            elif line:
                rows.append([int(x) for x in line.split()])
    lengths = [int(x) for x in meta["node_lengths"].split()]
    paths = [[int(x) for x in p.split()] for p in meta["paths"].split("|")]
    return np.array(rows, np.uint8), lengths, paths


def sdpa_masked(Q, K, V, mask, scale=None):
    """Dense masked attention via torch SDPA in fp64 (library routine).
    Q [T,Hq,D], K/V [T,Hkv,D]; mask [T,T] bool.  Returns O [T,Hq,D]."""
    Hq, Hkv = Q.shape[1], K.shape[1]
    g = Hq // Hkv
    q = Q.permute(1, 0, 2)[None]
    k = K.repeat_interleave(g, dim=1).permute(1, 0, 2)[None]
    v = V.repeat_interleave(g, dim=1).permute(1, 0, 2)[None]
    o = F.scaled_dot_product_attention(q, k, v, attn_mask=torch.as_tensor(mask, dtype=torch.bool), scale=scale)
    return o[0].permute(1, 0, 2)


def causal_sdpa(Q, K, V):
    Hq, Hkv = Q.shape[1], K.shape[1]
    g = Hq // Hkv
    q = Q.permute(1, 0, 2)[None]
    k = K.repeat_interleave(g, dim=1).permute(1, 0, 2)[None]
    v = V.repeat_interleave(g, dim=1).permute(1, 0, 2)[None]
    return F.scaled_dot_product_attention(q, k, v, is_causal=True)[0].permute(1, 0, 2)


def rand_qkv(T, Hq, Hkv, D, seed):
    g = torch.Generator().manual_seed(seed)
    return tuple(torch.randn(T, h, D, generator=g, dtype=torch.float64) for h in (Hq, Hkv, Hkv, Hq))


def random_grpo_specs(rng, n_groups, max_p=20, max_g=4, max_r=9):
    specs = []
    for _ in range(n_groups):
        P = int(rng.integers(0, max_p + 1))
        G = int(rng.integers(1, max_g + 1))
        specs.append((P, [int(rng.integers(1, max_r + 1)) for _ in range(G)]))
    return specs


# ---------------------------------------------------------------------------
# mask
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["mask_grpo_P2_R2_R1.txt", "mask_tree_depth3.txt", "mask_docs_2_3.txt"])
def test_mask_hand_written(name):
    want, lengths, paths = read_golden_mask(name)
    st = W.tree_structure(lengths, paths)
    got = orc.dense_mask(orc.structure_labels(st))
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("seed", range(12))
def test_mask_equals_segment_rule(seed):
    rng = np.random.default_rng(seed)
    st = W.grpo_structure(random_grpo_specs(rng, int(rng.integers(1, 4))))
    want = p2_mask_mod(st.group_id, st.suffix_id)
    np.testing.assert_array_equal(orc.dense_mask(orc.structure_labels(st)), want)
    np.testing.assert_array_equal(orc.dense_mask(orc.seg_labels(st.group_id, st.suffix_id)), want)


def test_mask_docs_block_causal():
    lengths = [3, 1, 5, 2]
    st = W.docs_structure(lengths)
    T = sum(lengths)
    want = np.zeros((T, T), np.uint8)
    o = 0
    for n in lengths:
        want[o:o + n, o:o + n] = np.tril(np.ones((n, n), np.uint8))
        o += n
    np.testing.assert_array_equal(orc.dense_mask(orc.structure_labels(st)), want)
    np.testing.assert_array_equal(orc.dense_mask(orc.seg_labels(st.group_id, st.suffix_id)), want)


def test_useful_pairs_closed_form():
    # per group: P(P+1)/2 + sum_i [R_i P + R_i (R_i + 1) / 2]
    for c in (1, 2, 3):
        st = W.config_structure(c)
        want = sum(P * (P + 1) // 2 + sum(R * P + R * (R + 1) // 2 for R in Rs) for P, Rs in st.meta["group_specs"])
        assert orc.count_pairs(orc.structure_labels(st)) == want


@pytest.mark.parametrize("bad", [
    dict(lengths=[2, 2], paths=[[1, 0]]),            # child before parent
    dict(lengths=[2, 2, 2], paths=[[0, 1], [0, 2], [1, 2]]),  # inconsistent parents
    dict(lengths=[2, 2, 2], paths=[[0, 1]]),         # node 2 on no path
    dict(lengths=[2, -1], paths=[[0, 1]]),           # negative length
    dict(lengths=[2, 2], paths=[[0, 5]]),            # node out of range
    dict(lengths=[2, 2], paths=[[0, 1], []]),        # empty path
])
def test_invalid_tree_rejected(bad):
    st = W.tree_structure(bad["lengths"], bad["paths"])
    with pytest.raises(orc.OracleError):
        orc.structure_labels(st)


@pytest.mark.parametrize("g,s", [
    ([0, 0, 0, 0], [1, 1, -1, -1]),      # prompt after a completion
    ([0, 0, 1, 1, 0], [-1, -1, -1, -1, -1]),  # group 0 not contiguous
    ([0, 0, 0, 1, 1], [-1, 3, 3, 4, 3]),  # completion id 3 reused
    ([0, 0, 0], [-1, 2, -1]),            # two prompt runs in a group
])
def test_invalid_segments_rejected(g, s):
    with pytest.raises(orc.OracleError):
        orc.seg_labels(g, s)


# ---------------------------------------------------------------------------
# block map
# ---------------------------------------------------------------------------

def tiles_by_numpy(mask, BM, BN):
    """Independent tiling of a dense mask: kinds[nq, nk]."""
    T = mask.shape[0]
    nq, nk = -(-T // BM), -(-T // BN)
    pad = np.zeros((nq * BM, nk * BN), np.int64)
    pad[:T, :T] = mask
    kept = pad.reshape(nq, BM, nk, BN).sum(axis=(1, 3))
    inr = np.zeros_like(pad)
    inr[:T, :T] = 1
    inrange = inr.reshape(nq, BM, nk, BN).sum(axis=(1, 3))
    return np.where(kept == 0, 0, np.where((kept == BM * BN) & (inrange == BM * BN), 1, 2)).astype(np.uint8)


def check_bm_against_kinds(bm, kinds):
    nq, nk = kinds.shape
    for i in range(nq):
        js = np.nonzero(kinds[i])[0]
        row = slice(bm["q_ptr"][i], bm["q_ptr"][i + 1])
        np.testing.assert_array_equal(bm["kv_idx"][row], js)
        np.testing.assert_array_equal(bm["kind"][row], kinds[i, js])
    for j in range(nk):
        is_ = np.nonzero(kinds[:, j])[0]
        col = slice(bm["k_ptr"][j], bm["k_ptr"][j + 1])
        np.testing.assert_array_equal(bm["q_idx"][col], is_)
        np.testing.assert_array_equal(bm["kindT"][col], kinds[is_, j])


@pytest.mark.parametrize("seed", range(10))
@pytest.mark.parametrize("BM,BN", [(16, 16), (32, 16), (16, 64), (128, 128)])
def test_blockmap_brute_force(seed, BM, BN):
    rng = np.random.default_rng(100 + seed)
    st = W.random_tree(rng, n_nodes=int(rng.integers(1, 12)), max_len=int(rng.integers(1, 90)))
    lab = orc.structure_labels(st)
    if lab.T == 0:
        return
    kinds = tiles_by_numpy(p2_like_tree_mask(st), BM, BN)
    check_bm_against_kinds(orc.blockmap(lab, BM, BN), kinds)


def p2_like_tree_mask(st):
    """Independent dense keep for a general tree: expand each token's
    ancestor-or-self node set by walking the sample paths."""
    T = st.T
    starts = np.concatenate([[0], np.cumsum(st.node_lengths)[:-1]]).astype(int)
    anc = {}
    for p in st.paths():
        for k, n in enumerate(p):
            anc[n] = set(p[: k + 1])
    node_of = np.repeat(np.arange(st.n_nodes), st.node_lengths)
    m = np.zeros((T, T), np.uint8)
    for q in range(T):
        for a in anc[node_of[q]]:
            s, e = starts[a], starts[a] + st.node_lengths[a]
            m[q, s:min(e, q + 1)] = 1
    return m


def test_blockmap_hand_written():
    with open(os.path.join(GOLDEN, "blockmap_grpo_aligned.txt")) as f:
        lines = [l.strip() for l in f if l.strip()]
    meta = {l[1:].partition(":")[0].strip(): l[1:].partition(":")[2].strip() for l in lines if l.startswith("#") and ":" in l}
    lengths = [int(x) for x in meta["node_lengths"].split()]
    paths = [[int(x) for x in p.split()] for p in meta["paths"].split("|")]
    BM, BN = (int(x) for x in meta["block"].split())
    bm = orc.blockmap(orc.structure_labels(W.tree_structure(lengths, paths)), BM, BN)
    rows = [l for l in lines if not l.startswith("#")]
    assert len(rows) == bm["nq"]
    for line in rows:
        i, _, rest = line.partition(":")
        i = int(i)
        ent = [(int(a), {"F": 1, "P": 2}[b]) for a, b in (e.split("/") for e in rest.split())]
        sl = slice(bm["q_ptr"][i], bm["q_ptr"][i + 1])
        assert list(zip(bm["kv_idx"][sl].tolist(), bm["kind"][sl].tolist())) == ent


@pytest.mark.parametrize("seed", range(4))
def test_blockmap_aligned_closed_form(seed):
    """Node lengths multiples of the tile B: tile (i, j) is full when node(j)
    is a proper ancestor of node(i) or j < i inside the same node, partial on
    the diagonal, empty otherwise."""
    rng = np.random.default_rng(7 + seed)
    B = 16
    st = W.random_tree(rng, n_nodes=int(rng.integers(2, 9)), max_len=4)
    st.node_lengths = st.node_lengths * B
    lab = orc.structure_labels(st)
    if lab.T == 0:
        return
    nt = lab.T // B
    tile_node = np.repeat(np.arange(st.n_nodes), st.node_lengths // B)
    parent = {}
    for p in st.paths():
        for a, b in zip(p[:-1], p[1:]):
            parent[b] = a

    def proper_anc(n):
        out = set()
        while n in parent:
            n = parent[n]
            out.add(n)
        return out

    kinds = np.zeros((nt, nt), np.uint8)
    for i in range(nt):
        for j in range(nt):
            if tile_node[j] in proper_anc(tile_node[i]) or (tile_node[j] == tile_node[i] and j < i):
                kinds[i, j] = 1
            elif i == j:
                kinds[i, j] = 2
    check_bm_against_kinds(orc.blockmap(lab, B, B), kinds)


def test_blockmap_workload1_counts():
    bm = orc.blockmap(orc.structure_labels(W.config_structure(1)), 16, 16)
    assert bm["nnz"] == 5 and int((bm["kind"] == 1).sum()) == 2 and int((bm["kind"] == 2).sum()) == 3


# ---------------------------------------------------------------------------
# forward
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(6))
def test_fwd_vs_sdpa_dense_mask(seed):
    rng = np.random.default_rng(seed)
    st = W.grpo_structure(random_grpo_specs(rng, 2))
    T = st.T
    Hq, Hkv, D = [(2, 1, 8), (4, 2, 16), (3, 3, 5)][seed % 3]
    Q, K, V, _ = rand_qkv(T, Hq, Hkv, D, seed)
    want = sdpa_masked(Q, K, V, p2_mask_mod(st.group_id, st.suffix_id))
    O, L = orc.attn_fwd(Q, K, V, orc.structure_labels(st))
    np.testing.assert_allclose(O, want.numpy(), rtol=0, atol=1e-12)


def test_fwd_tree_vs_sdpa_dense_mask():
    rng = np.random.default_rng(3)
    for _ in range(5):
        st = W.random_tree(rng, n_nodes=9, max_len=7)
        if st.T == 0:
            continue
        Q, K, V, _ = rand_qkv(st.T, 4, 2, 8, 11)
        want = sdpa_masked(Q, K, V, p2_like_tree_mask(st))
        O, _ = orc.attn_fwd(Q, K, V, orc.structure_labels(st))
        np.testing.assert_allclose(O, want.numpy(), rtol=0, atol=1e-12)


def unfolded_sequences(st):
    """For every node, the token indices of [ancestors...; own node] in order."""
    starts = np.concatenate([[0], np.cumsum(st.node_lengths)[:-1]]).astype(int)
    seqs = {}
    for p in st.paths():
        for k, n in enumerate(p):
            seqs[n] = np.concatenate([np.arange(starts[a], starts[a] + st.node_lengths[a]) for a in p[: k + 1]])
    return starts, seqs


@pytest.mark.parametrize("which", ["grpo", "tree", "docs"])
def test_fwd_unfolded_invariant(which):
    """Every token's output and LSE equal plain causal attention over the
    unfolded sequence [ancestor nodes...; own node], gathered at that token
    ("prefix_grouper_kernel.py": each suffix token attends to the single
    shared prefix plus causally within its own suffix)."""
    rng = np.random.default_rng(5)
    st = {"grpo": lambda: W.grpo_structure([(13, [5, 9, 1]), (0, [4, 6]), (7, [3])]),
          "tree": lambda: W.tree_structure([6, 3, 4, 2, 5, 3], [[0, 1, 2], [0, 1, 3], [0, 4, 5]]),
          "docs": lambda: W.docs_structure([5, 1, 8, 3])}[which]()
    Hq, Hkv, D = 4, 2, 8
    Q, K, V, _ = rand_qkv(st.T, Hq, Hkv, D, 21)
    O, L = orc.attn_fwd(Q, K, V, orc.structure_labels(st))
    starts, seqs = unfolded_sequences(st)
    D_ = Q.shape[2]
    for n, idx in seqs.items():
        ln = int(st.node_lengths[n])
        if ln == 0:
            continue
        sl = torch.as_tensor(idx)
        ref = causal_sdpa(Q[sl], K[sl], V[sl])
        # own node's tokens are the last ln of the unfolded sequence
        np.testing.assert_allclose(O[starts[n]:starts[n] + ln], ref[-ln:].numpy(), rtol=0, atol=1e-12)
        # LSE: log-sum-exp of the unfolded causal scores
        s = torch.einsum("thd,uhd->htu", Q[sl], K[sl].repeat_interleave(Hq // Hkv, dim=1)) / np.sqrt(D_)
        s = s.masked_fill(~torch.ones(len(idx), len(idx), dtype=torch.bool).tril(), float("-inf"))
        lse = torch.logsumexp(s, dim=-1)[:, -ln:]
        np.testing.assert_allclose(L[:, starts[n]:starts[n] + ln], lse.numpy(), rtol=0, atol=1e-12)


def test_fwd_uniform_v():
    st = W.config_structure(1)
    Q, K, V, _ = rand_qkv(st.T, 2, 2, 32, 4)
    v0 = torch.randn(2, 32, dtype=torch.float64)
    V = v0[None].expand(st.T, 2, 32).contiguous()
    O, _ = orc.attn_fwd(Q, K, V, orc.structure_labels(st))
    np.testing.assert_allclose(O, np.broadcast_to(v0.numpy()[None], O.shape), rtol=0, atol=1e-13)


def test_fwd_one_token_suffix_isolated():
    """A one-token completion attends to prompt + itself only: changing the
    other completions' K/V leaves its output unchanged."""
    st = W.grpo_structure([(6, [3, 1, 4])])
    lab = orc.structure_labels(st)
    Q, K, V, _ = rand_qkv(st.T, 2, 1, 8, 9)
    t = 6 + 3  # the one-token completion
    O1, L1 = orc.attn_fwd(Q, K, V, lab, rows=[t])
    K2, V2 = K.clone(), V.clone()
    K2[6:9] += 3.0
    V2[10:] -= 2.0
    O2, L2 = orc.attn_fwd(Q, K2, V2, lab, rows=[t])
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)
    # and it equals softmax over prompt + self
    idx = torch.as_tensor(list(range(6)) + [t])
    ref = causal_sdpa(Q[idx], K[idx], V[idx])[-1]
    np.testing.assert_allclose(O1[0], ref.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("specs", [[(0, [17])], [(0, [5, 9, 3])], [(23, [])]])
def test_fwd_degenerate_is_textbook_causal(specs):
    """P = 0 (each completion alone) and a bare prompt are plain causal attention."""
    st = W.grpo_structure(specs)
    Q, K, V, _ = rand_qkv(st.T, 2, 2, 8, 1)
    O, _ = orc.attn_fwd(Q, K, V, orc.structure_labels(st))
    o = 0
    for n in st.node_lengths:
        n = int(n)
        if n:
            ref = causal_sdpa(Q[o:o + n], K[o:o + n], V[o:o + n])
            np.testing.assert_allclose(O[o:o + n], ref.numpy(), rtol=0, atol=1e-12)
        o += n


def test_fwd_single_completion_is_causal():
    """G = 1: prompt + one completion is ordinary causal attention."""
    st = W.grpo_structure([(9, [7])])
    Q, K, V, _ = rand_qkv(st.T, 2, 1, 8, 2)
    O, _ = orc.attn_fwd(Q, K, V, orc.structure_labels(st))
    np.testing.assert_allclose(O, causal_sdpa(Q, K, V).numpy(), rtol=0, atol=1e-12)


def test_fwd_rows_subset_and_row_sum():
    st = W.grpo_structure([(11, [4, 7]), (5, [3, 3])])
    lab = orc.structure_labels(st)
    Q, K, V, _ = rand_qkv(st.T, 4, 2, 8, 3)
    O, L = orc.attn_fwd(Q, K, V, lab)
    rows = [0, 5, st.T - 1, 13]
    Os, Ls = orc.attn_fwd(Q, K, V, lab, rows=rows)
    np.testing.assert_array_equal(Os, O[rows])
    np.testing.assert_array_equal(Ls, L[:, rows])
    # softmax rows sum to one: sum_kv mask * exp(s - LSE) == 1
    m = p2_mask_mod(st.group_id, st.suffix_id).astype(bool)
    s = np.einsum("thd,uhd->htu", Q.numpy(), K.numpy().repeat(2, axis=1)) / np.sqrt(8)
    tot = np.where(m[None], np.exp(s - L[:, :, None]), 0.0).sum(-1)
    np.testing.assert_allclose(tot, 1.0, rtol=0, atol=1e-13)


def test_fwd_custom_scale():
    st = W.grpo_structure([(5, [4, 2])])
    Q, K, V, _ = rand_qkv(st.T, 2, 2, 8, 6)
    want = sdpa_masked(Q, K, V, p2_mask_mod(st.group_id, st.suffix_id), scale=0.3)
    O, _ = orc.attn_fwd(Q, K, V, orc.structure_labels(st), scale=0.3)
    np.testing.assert_allclose(O, want.numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# backward
# ---------------------------------------------------------------------------

def autograd_grads(Q, K, V, dO, mask, scale=None):
    Q, K, V = (x.clone().requires_grad_(True) for x in (Q, K, V))
    O = sdpa_masked(Q, K, V, mask, scale=scale)
    O.backward(dO)
    return Q.grad.numpy(), K.grad.numpy(), V.grad.numpy()


@pytest.mark.parametrize("seed", range(5))
def test_bwd_vs_autograd(seed):
    rng = np.random.default_rng(40 + seed)
    if seed % 2:
        st = W.random_tree(rng, n_nodes=8, max_len=6)
        mask = p2_like_tree_mask(st)
    else:
        st = W.grpo_structure(random_grpo_specs(rng, 2))
        mask = p2_mask_mod(st.group_id, st.suffix_id)
    if st.T == 0:
        return
    Hq, Hkv, D = [(2, 1, 8), (4, 2, 6), (3, 3, 4)][seed % 3]
    Q, K, V, dO = rand_qkv(st.T, Hq, Hkv, D, seed)
    dq, dk, dv = orc.attn_bwd(Q, K, V, dO, orc.structure_labels(st))
    wq, wk, wv = autograd_grads(Q, K, V, dO, mask)
    np.testing.assert_allclose(dq, wq, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, wk, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, wv, rtol=0, atol=1e-11)


def test_bwd_finite_differences():
    """Central differences of L = sum dO * O, using the oracle's own forward."""
    st = W.grpo_structure([(4, [3, 2])])
    lab = orc.structure_labels(st)
    Q, K, V, dO = rand_qkv(st.T, 2, 1, 4, 17)
    dq, dk, dv = orc.attn_bwd(Q, K, V, dO, lab)
    eps = 1e-6

    def loss(q, k, v):
        O, _ = orc.attn_fwd(q, k, v, lab)
        return float((O * dO.numpy()).sum())

    rng = np.random.default_rng(0)
    for name, X, G in (("Q", Q, dq), ("K", K, dk), ("V", V, dv)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, s)) for s in X.shape)
            xp, xm = X.clone(), X.clone()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = [Q, K, V]
            args_m = [Q, K, V]
            pos = "QKV".index(name)
            args_p[pos], args_m[pos] = xp, xm
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - G[idx]) < 1e-7, (name, idx, fd, G[idx])


def test_bwd_sum_invariants():
    """sum_j dS_ij = 0 for every row, so dK summed over all kv tokens is 0 per
    kv head; and sum_j P_ij = 1, so dV summed over all kv tokens equals dO
    summed over rows and the kv head's q heads."""
    st = W.config_structure(1)
    Q, K, V, dO = rand_qkv(st.T, 4, 2, 8, 5)
    _, dk, dv = orc.attn_bwd(Q, K, V, dO, orc.structure_labels(st))
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12)
    want = dO.numpy().reshape(st.T, 2, 2, 8).sum(axis=(0, 2))
    np.testing.assert_allclose(dv.sum(axis=0), want, atol=1e-12)


def test_bwd_unfolded_invariant():
    """Unfold a group into one causal sequence per completion, give the prompt
    rows' upstream gradient to copy 0 only: the prompt's dK/dV are the sums
    over copies, completion rows match row for row, and the prompt's dQ is
    copy 0's."""
    P, Rs = 6, [4, 3, 5]
    st = W.grpo_structure([(P, Rs)])
    Q, K, V, dO = rand_qkv(st.T, 2, 1, 8, 33)
    dq, dk, dv = orc.attn_bwd(Q, K, V, dO, orc.structure_labels(st))
    sum_dk = np.zeros((P, 1, 8))
    sum_dv = np.zeros((P, 1, 8))
    o = P
    for c, R in enumerate(Rs):
        idx = torch.as_tensor(list(range(P)) + list(range(o, o + R)))
        q, k, v = (x[idx].clone().requires_grad_(True) for x in (Q, K, V))
        g = dO[idx].clone()
        if c > 0:
            g[:P] = 0
        causal_sdpa(q, k, v).backward(g)
        np.testing.assert_allclose(dq[o:o + R], q.grad[P:].numpy(), atol=1e-12)
        np.testing.assert_allclose(dk[o:o + R], k.grad[P:].numpy(), atol=1e-12)
        np.testing.assert_allclose(dv[o:o + R], v.grad[P:].numpy(), atol=1e-12)
        if c == 0:
            np.testing.assert_allclose(dq[:P], q.grad[:P].numpy(), atol=1e-12)
        sum_dk += k.grad[:P].numpy()
        sum_dv += v.grad[:P].numpy()
        o += R
    np.testing.assert_allclose(dk[:P], sum_dk, atol=1e-12)
    np.testing.assert_allclose(dv[:P], sum_dv, atol=1e-12)


def test_bwd_subsets_match_full():
    st = W.grpo_structure([(9, [4, 6]), (3, [5])])
    lab = orc.structure_labels(st)
    Q, K, V, dO = rand_qkv(st.T, 4, 2, 8, 8)
    dq, dk, dv = orc.attn_bwd(Q, K, V, dO, lab)
    rows, cols = [0, 7, 12, st.T - 1], [1, 9, 14, st.T - 2]
    sq, sk, sv = orc.attn_bwd(Q, K, V, dO, lab, qrows=rows, kvcols=cols)
    np.testing.assert_allclose(sq, dq[rows], atol=1e-13)
    np.testing.assert_allclose(sk, dk[cols], atol=1e-13)
    np.testing.assert_allclose(sv, dv[cols], atol=1e-13)
