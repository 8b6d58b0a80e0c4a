"""Seeded synthetic workloads for prefix-tree attention.

This module only *describes* inputs: tree structures (node lengths plus
root-to-leaf sample paths), the equivalent per-token segment labels for the
shared-prefix (GRPO) and packed-document cases, and N(0,1) tensors drawn from
fixed seeds.  It holds none of the attention arithmetic and none of the mask
rule, so both the fp64 oracle and the CUDA path can consume it.

Workload shapes follow the pages' settings:

* GRPO shared-prefix groups: one prompt of P tokens followed by G completions
  ("cp=1 shared-prefix prefix-tree attention for rollouts", PR description;
  "prefix_grouper_kernel.py", ``build_seg_info_multigroup``).
* A general prefix tree given as ``(node_lengths, sample_paths)``
  ("cp=1 shared-prefix prefix-tree attention for rollouts", ``AttnMaskSpec.prefix_tree``).
* Packed documents, i.e. a forest of single-node trees (the doc-gated,
  block-causal mask of "support sequence packing in the Domino and JetSpec drafts").
* Draft blocks (DFlash): a packed context of documents and one block of
  ``block_size`` tokens per anchor, anchors drawn so that a whole block stays
  inside its document ("support sequence packing in the Domino and JetSpec
  drafts": anchor sampling keeps doc_remaining >= block_size - 1).

Lengths come from ``numpy.random.default_rng(seed)`` with inclusive integer
draws; tensors from a CPU ``torch.Generator`` seeded ``1000 + seed`` in fp32,
then cast, so every consumer sees identical values.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import numpy as np

__all__ = [
    "Structure",
    "DraftStructure",
    "grpo_structure",
    "tree_structure",
    "docs_structure",
    "random_tree",
    "CONFIGS",
    "config_structure",
    "make_tensors",
]


@dataclass
class Structure:
    """A prefix tree laid out flat.

    node_lengths[i] tokens of node i sit contiguously, nodes in id order.
    path_ptr/path_nodes is a CSR list of root->leaf paths (one per sample).
    group_id/suffix_id are the equivalent segment labels when the tree has
    depth <= 2 (prefix node = suffix_id -1); None for deeper trees.
    """

    node_lengths: np.ndarray  # int32 [n_nodes]
    path_ptr: np.ndarray  # int32 [n_samples + 1]
    path_nodes: np.ndarray  # int32 [path_ptr[-1]]
    group_id: Optional[np.ndarray] = None  # int32 [T]
    suffix_id: Optional[np.ndarray] = None  # int32 [T]
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return int(self.node_lengths.sum()) if self.node_lengths.size else 0

    @property
    def n_nodes(self) -> int:
        return int(self.node_lengths.size)

    @property
    def n_samples(self) -> int:
        return int(self.path_ptr.size - 1)

    def paths(self) -> List[List[int]]:
        return [
            [int(x) for x in self.path_nodes[self.path_ptr[s] : self.path_ptr[s + 1]]]
            for s in range(self.n_samples)
        ]


def _csr(paths: Sequence[Sequence[int]]) -> Tuple[np.ndarray, np.ndarray]:
    ptr = np.zeros(len(paths) + 1, dtype=np.int32)
    for i, p in enumerate(paths):
        ptr[i + 1] = ptr[i] + len(p)
    nodes = np.array([n for p in paths for n in p], dtype=np.int32)
    return ptr, nodes


def grpo_structure(group_specs: Sequence[Tuple[int, Sequence[int]]], name: str = "") -> Structure:
    """Groups packed flat as ``[prompt_g | c_g0 | c_g1 | ...]`` for g = 0, 1, ...

    ``group_specs`` is a list of ``(P_g, [R_g0, R_g1, ...])``.  The tree form
    gives each group a prompt node (possibly of length 0) followed by one
    node per completion; each sample path is ``[prompt, completion]``.  The
    segment form labels every token with its group and, for completion
    tokens, a globally unique completion id (-1 on prompt tokens).
    """
    lengths: List[int] = []
    paths: List[List[int]] = []
    gid: List[np.ndarray] = []
    sid: List[np.ndarray] = []
    suffix_counter = 0
    for g, (P, Rs) in enumerate(group_specs):
        root = len(lengths)
        lengths.append(int(P))
        gid.append(np.full(int(P), g, dtype=np.int32))
        sid.append(np.full(int(P), -1, dtype=np.int32))
        for r in Rs:
            node = len(lengths)
            lengths.append(int(r))
            paths.append([root, node])
            gid.append(np.full(int(r), g, dtype=np.int32))
            sid.append(np.full(int(r), suffix_counter, dtype=np.int32))
            suffix_counter += 1
        if len(Rs) == 0:
            paths.append([root])
    ptr, nodes = _csr(paths)
    return Structure(
        node_lengths=np.asarray(lengths, dtype=np.int32),
        path_ptr=ptr,
        path_nodes=nodes,
        group_id=np.concatenate(gid) if gid else np.zeros(0, np.int32),
        suffix_id=np.concatenate(sid) if sid else np.zeros(0, np.int32),
        name=name,
        meta={"group_specs": [(int(P), [int(r) for r in Rs]) for P, Rs in group_specs]},
    )


def docs_structure(doc_lengths: Sequence[int], name: str = "") -> Structure:
    """Packed documents: every document is a one-node tree (its own group,
    prompt-only in the segment form, so it is plain causal inside)."""
    lengths = [int(x) for x in doc_lengths]
    paths = [[i] for i in range(len(lengths))]
    ptr, nodes = _csr(paths)
    gid = np.concatenate([np.full(n, i, np.int32) for i, n in enumerate(lengths)]) if lengths else np.zeros(0, np.int32)
    sid = np.full(int(sum(lengths)), -1, dtype=np.int32)
    return Structure(
        node_lengths=np.asarray(lengths, dtype=np.int32),
        path_ptr=ptr,
        path_nodes=nodes,
        group_id=gid,
        suffix_id=sid,
        name=name,
        meta={"doc_lengths": lengths},
    )


def tree_structure(node_lengths: Sequence[int], paths: Sequence[Sequence[int]], name: str = "") -> Structure:
    ptr, nodes = _csr(paths)
    return Structure(
        node_lengths=np.asarray([int(x) for x in node_lengths], dtype=np.int32),
        path_ptr=ptr,
        path_nodes=nodes,
        name=name,
    )


def random_tree(rng: np.random.Generator, n_nodes: int, max_len: int, p_zero: float = 0.1,
                max_depth: int = 4) -> Structure:
    """A random prefix tree laid out in DFS order (every parent precedes its
    children), with some zero-length nodes.  Used for small brute-force checks."""
    parent = [-1]
    depth = [0]
    # grow: each new node hangs under a random existing node (bounded depth), then
    # relabel in DFS order so ids are contiguous per subtree.
    for i in range(1, n_nodes):
        while True:
            p = int(rng.integers(-1, i))  # -1 = new root
            if p == -1 or depth[p] + 1 < max_depth:
                break
        parent.append(p)
        depth.append(0 if p == -1 else depth[p] + 1)
    children: List[List[int]] = [[] for _ in range(n_nodes)]
    roots = []
    for i, p in enumerate(parent):
        (roots if p == -1 else children[p]).append(i)
    order: List[int] = []
    stack = list(reversed(roots))
    while stack:
        u = stack.pop()
        order.append(u)
        stack.extend(reversed(children[u]))
    new_id = {u: k for k, u in enumerate(order)}
    lengths = [0] * n_nodes
    for u in order:
        ln = 0 if rng.random() < p_zero else int(rng.integers(1, max_len + 1))
        lengths[new_id[u]] = ln
    # one path per leaf: root -> leaf
    paths = []
    for u in order:
        if not children[u]:
            chain = []
            v = u
            while v != -1:
                chain.append(new_id[v])
                v = parent[v]
            paths.append(chain[::-1])
    return tree_structure(lengths, paths, name="random_tree")


# ---------------------------------------------------------------------------
@dataclass
class DraftStructure:
    """A draft-block layout: ctx_len context tokens, then one block of
    block_size tokens per anchor (block b's token k at real position
    anchors[b] + k); ctx_doc / anchor_doc are the packed documents of the
    context tokens and of the anchors."""

    ctx_len: int
    anchors: np.ndarray  # int32 [n_blocks]
    block_size: int
    block_keep: Optional[np.ndarray] = None  # bool [n_blocks], None: all kept
    causal: bool = False
    window: int = 0
    ctx_doc: Optional[np.ndarray] = None  # int32 [ctx_len]
    anchor_doc: Optional[np.ndarray] = None  # int32 [n_blocks]
    name: str = ""

    @property
    def T(self) -> int:
        return int(self.ctx_len + self.anchors.size * self.block_size)

    def kwargs(self) -> dict:
        """The layout as keyword arguments (the draft map builder and the oracle take the same names)."""
        return dict(ctx_len=self.ctx_len, anchors=self.anchors, block_size=self.block_size,
                    block_keep=self.block_keep, causal=self.causal, window=self.window,
                    ctx_doc=self.ctx_doc, anchor_doc=self.anchor_doc)


def draft_structure(rng: np.random.Generator, ctx_len: int, doc_min: int, doc_max: int, n_blocks: int,
                    block_size: int, causal: bool = False, window: int = 0, name: str = "") -> DraftStructure:
    """Context packed with documents U[doc_min, doc_max] (the last cut to fill
    it); n_blocks anchors drawn without replacement from the positions whose
    whole block stays inside the document, sorted."""
    docs: List[int] = []
    left = ctx_len
    while left > 0:
        d = min(int(rng.integers(doc_min, doc_max + 1)), left)
        docs.append(d)
        left -= d
    ctx_doc = np.repeat(np.arange(len(docs), dtype=np.int32), docs)
    ends = np.cumsum(docs)
    doc_end = ends[ctx_doc]
    valid = np.nonzero(doc_end - np.arange(ctx_len) >= block_size)[0]
    anchors = np.sort(rng.choice(valid, size=n_blocks, replace=False)).astype(np.int32)
    return DraftStructure(ctx_len=ctx_len, anchors=anchors, block_size=block_size, causal=causal, window=window,
                          ctx_doc=ctx_doc, anchor_doc=ctx_doc[anchors].astype(np.int32), name=name)


# The reference workloads (synthetic, seeded)
# ---------------------------------------------------------------------------

CONFIGS = {
    1: dict(name="tiny shared-prefix GRPO: 1 group, P=16, G=4 x R=8 (T=48), Hq=Hkv=2, D=32, fp32",
            Hq=2, Hkv=2, D=32, dtype="f32"),
    2: dict(name="GRPO batch: 8 groups, P=512, G=8, R~U[64,256], Hq=14, Hkv=2, D=64, bf16",
            Hq=14, Hkv=2, D=64, dtype="bf16"),
    3: dict(name="long-prompt GRPO: 2 groups, P=4096, G=16, R~U[256,1024], Hq=32, Hkv=8, D=128, bf16",
            Hq=32, Hkv=8, D=128, dtype="bf16"),
    4: dict(name="depth-3 prefix tree: root 1024 -> 4 x 512 -> 4 x U[128,384] each, Hq=16, Hkv=4, D=128, bf16",
            Hq=16, Hkv=4, D=128, dtype="bf16"),
    5: dict(name="packed documents: 4 rows x 4096, docs U[64,2048] cut to fill the row, Hq=8, Hkv=2, D=256, bf16",
            Hq=8, Hkv=2, D=256, dtype="bf16"),
    6: dict(name="DFlash draft blocks: context 4096 packed with docs U[256,2048], 256 in-document blocks of 16, "
                 "bidirectional, document-gated, Hq=16, Hkv=4, D=128, bf16",
            Hq=16, Hkv=4, D=128, dtype="bf16", kind="draft"),
    7: dict(name="packed documents at head_dim 512: 4 rows x 4096, docs U[64,2048] cut to fill the row, "
                 "Hq=8, Hkv=2, D=512, bf16",
            Hq=8, Hkv=2, D=512, dtype="bf16"),
}


def config_structure(c: int):
    """The token layout of workload ``c`` (1..7), lengths drawn from default_rng(c): a
    Structure, or a DraftStructure for the draft-block workload."""
    rng = np.random.default_rng(c)
    if c == 1:
        return grpo_structure([(16, [8, 8, 8, 8])], name="c1")
    if c == 2:
        specs = [(512, [int(x) for x in rng.integers(64, 256 + 1, size=8)]) for _ in range(8)]
        return grpo_structure(specs, name="c2")
    if c == 3:
        specs = [(4096, [int(x) for x in rng.integers(256, 1024 + 1, size=16)]) for _ in range(2)]
        return grpo_structure(specs, name="c3")
    if c == 4:
        lengths = [1024]
        paths = []
        for _ in range(4):
            child = len(lengths)
            lengths.append(512)
            for _ in range(4):
                leaf = len(lengths)
                lengths.append(int(rng.integers(128, 384 + 1)))
                paths.append([0, child, leaf])
        return tree_structure(lengths, paths, name="c4")
    if c in (5, 7):
        docs: List[int] = []
        for _ in range(4):
            left = 4096
            while left > 0:
                d = int(rng.integers(64, 2048 + 1))
                d = min(d, left)
                docs.append(d)
                left -= d
        return docs_structure(docs, name=f"c{c}")
    if c == 6:
        return draft_structure(rng, 4096, 256, 2048, 256, 16, name="c6")
    raise ValueError(f"unknown workload {c}")


def make_tensors(T: int, Hq: int, Hkv: int, D: int, dtype: str, seed: int):
    """Q, K, V, dO ~ N(0,1): fp32 draws from a CPU generator seeded
    ``1000 + seed``, then cast to ``dtype`` ("f32" or "bf16").  Token-major
    layout: Q and dO are [T, Hq, D]; K and V are [T, Hkv, D]."""
    import torch

    g = torch.Generator(device="cpu").manual_seed(1000 + int(seed))
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]
    q = torch.randn(T, Hq, D, generator=g, dtype=torch.float32).to(tdt)
    k = torch.randn(T, Hkv, D, generator=g, dtype=torch.float32).to(tdt)
    v = torch.randn(T, Hkv, D, generator=g, dtype=torch.float32).to(tdt)
    do = torch.randn(T, Hq, D, generator=g, dtype=torch.float32).to(tdt)
    return q, k, v, do
