"""Python access to the fp64 C oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg may import this module; the library and its binding never do.

Every function takes and returns numpy arrays.  Floating-point inputs are
widened to fp64 exactly (bf16 and fp32 values are representable in fp64), so
the oracle sees precisely the values the GPU path sees.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OR_OK = 0


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (plain -O2, no arch flags)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
            u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")
            f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
            vp = ctypes.c_void_p
            lib.or_tree_labels.argtypes = [ctypes.c_int32, i32p, ctypes.c_int32, i32p, i32p, i32p, ctypes.c_int64, i32p]
            lib.or_seg_labels.argtypes = [ctypes.c_int64, i32p, i32p, i32p, i32p, ctypes.POINTER(ctypes.c_int32)]
            lib.or_dense_mask.argtypes = [ctypes.c_int64, i32p, i32p, u8p]
            lib.or_dense_mask.restype = None
            lib.or_count_pairs.argtypes = [ctypes.c_int64, i32p, i32p, ctypes.c_int]
            lib.or_count_pairs.restype = ctypes.c_int64
            lib.or_blockmap.argtypes = [ctypes.c_int64, i32p, i32p, ctypes.c_int32, ctypes.c_int32,
                                        i32p, i32p, u8p, i32p, i32p, u8p, ctypes.POINTER(ctypes.c_int64), ctypes.c_int]
            lib.or_attn_fwd.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                        f64p, f64p, f64p, i32p, i32p, ctypes.c_int64, vp, f64p, f64p, ctypes.c_int]
            lib.or_attn_bwd.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                        f64p, f64p, f64p, f64p, i32p, i32p,
                                        ctypes.c_int64, vp, vp, ctypes.c_int64, vp, vp, vp, ctypes.c_int]
            for f in ("or_tree_labels", "or_seg_labels", "or_blockmap", "or_attn_fwd", "or_attn_bwd"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


class OracleError(ValueError):
    pass


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _f64(a) -> np.ndarray:
    try:
        import torch

        if isinstance(a, torch.Tensor):
            a = a.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


class Labels:
    """Per-token node ids plus parent links: the prefix tree the oracle masks with."""

    def __init__(self, node_of: np.ndarray, parent: np.ndarray):
        self.node_of = _i32(node_of)
        self.parent = _i32(parent) if len(parent) else np.zeros(1, np.int32)
        self.T = int(self.node_of.size)


def tree_labels(node_lengths, path_ptr, path_nodes) -> Labels:
    """Labels from the tree form (node lengths + CSR sample paths)."""
    lib = _load()
    nl = _i32(node_lengths)
    pp = _i32(path_ptr)
    pn = _i32(path_nodes) if len(path_nodes) else np.zeros(1, np.int32)
    T = int(nl.sum()) if nl.size else 0
    parent = np.zeros(max(1, nl.size), np.int32)
    node_of = np.zeros(max(1, T), np.int32)
    rc = lib.or_tree_labels(int(nl.size), nl if nl.size else np.zeros(1, np.int32), int(pp.size - 1), pp, pn,
                            parent, T, node_of)
    if rc != OR_OK:
        raise OracleError(f"invalid tree (code {rc})")
    return Labels(node_of[:T], parent[: nl.size])


def seg_labels(group_id, suffix_id) -> Labels:
    """Labels from the segment form (per-token group id, suffix id; -1 = prompt)."""
    lib = _load()
    g = _i32(group_id)
    s = _i32(suffix_id)
    if g.shape != s.shape:
        raise OracleError("group_id and suffix_id differ in length")
    T = int(g.size)
    node_of = np.zeros(max(1, T), np.int32)
    parent = np.zeros(max(1, T), np.int32)
    n = ctypes.c_int32(0)
    rc = lib.or_seg_labels(T, g if T else np.zeros(1, np.int32), s if T else np.zeros(1, np.int32),
                           node_of, parent, ctypes.byref(n))
    if rc != OR_OK:
        raise OracleError(f"invalid segment labels (code {rc})")
    return Labels(node_of[:T], parent[: n.value])


def structure_labels(st) -> Labels:
    return tree_labels(st.node_lengths, st.path_ptr, st.path_nodes)


def dense_mask(lab: Labels) -> np.ndarray:
    """The T x T keep matrix (uint8).  Small T only."""
    lib = _load()
    T = lab.T
    m = np.zeros((max(T, 1), max(T, 1)), np.uint8)
    if T:
        lib.or_dense_mask(T, lab.node_of, lab.parent, m)
    return m[:T, :T]


def count_pairs(lab: Labels, n_threads: Optional[int] = None) -> int:
    """Kept (q, kv) pairs per head."""
    lib = _load()
    if lab.T == 0:
        return 0
    return int(lib.or_count_pairs(lab.T, lab.node_of, lab.parent, n_threads or default_threads()))


def blockmap(lab: Labels, BM: int, BN: int, n_threads: Optional[int] = None):
    """Brute-force block map.  Returns dict with q-major CSR (q_ptr, kv_idx,
    kind) and its kv-major transpose (k_ptr, q_idx, kindT); kind 1 = full,
    2 = partial."""
    lib = _load()
    T = lab.T
    nq = (T + BM - 1) // BM
    nk = (T + BN - 1) // BN
    cap = max(1, nq * nk)
    q_ptr = np.zeros(nq + 1, np.int32)
    k_ptr = np.zeros(nk + 1, np.int32)
    kv_idx = np.zeros(cap, np.int32)
    q_idx = np.zeros(cap, np.int32)
    kind = np.zeros(cap, np.uint8)
    kindT = np.zeros(cap, np.uint8)
    nnz = ctypes.c_int64(0)
    node_of = lab.node_of if T else np.zeros(1, np.int32)
    rc = lib.or_blockmap(T, node_of, lab.parent, BM, BN, q_ptr, kv_idx, kind, k_ptr, q_idx, kindT,
                         ctypes.byref(nnz), n_threads or default_threads())
    if rc != OR_OK:
        raise OracleError(f"blockmap failed (code {rc})")
    e = nnz.value
    return dict(q_ptr=q_ptr, kv_idx=kv_idx[:e], kind=kind[:e], k_ptr=k_ptr, q_idx=q_idx[:e], kindT=kindT[:e],
                nnz=e, nq=nq, nk=nk)


def attn_fwd(Q, K, V, lab: Labels, scale: float = 0.0, rows=None, n_threads: Optional[int] = None
             ) -> Tuple[np.ndarray, np.ndarray]:
    """fp64 forward.  Q [T,Hq,D], K/V [T,Hkv,D].  Returns O [n,Hq,D] and
    LSE [Hq,n] over ``rows`` (default: all T rows).  scale <= 0 means 1/sqrt(D)."""
    lib = _load()
    Qd, Kd, Vd = _f64(Q), _f64(K), _f64(V)
    T, Hq, D = Qd.shape
    Hkv = Kd.shape[1]
    if rows is None:
        n, rp = T, None
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n, rp = int(r.size), r.ctypes.data_as(ctypes.c_void_p)
    O = np.zeros((max(n, 1), Hq, D), np.float64)
    L = np.zeros((Hq, max(n, 1)), np.float64)
    rc = lib.or_attn_fwd(T, Hq, Hkv, D, float(scale), Qd, Kd, Vd, lab.node_of if T else np.zeros(1, np.int32),
                         lab.parent, n, rp, O, L, n_threads or default_threads())
    if rc != OR_OK:
        raise OracleError(f"attn_fwd failed (code {rc})")
    return O[:n], np.ascontiguousarray(L[:, :n])


def attn_bwd(Q, K, V, dO, lab: Labels, scale: float = 0.0, qrows=None, kvcols=None,
             n_threads: Optional[int] = None, want_dq: bool = True, want_dkv: bool = True):
    """fp64 backward.  Returns (dQ [nq_rows,Hq,D] or None, dK [n_cols,Hkv,D] or None,
    dV [n_cols,Hkv,D] or None) over the requested rows/columns (default all)."""
    lib = _load()
    Qd, Kd, Vd, dOd = _f64(Q), _f64(K), _f64(V), _f64(dO)
    T, Hq, D = Qd.shape
    Hkv = Kd.shape[1]

    def sel(a):
        if a is None:
            return T, None, None
        arr = np.ascontiguousarray(np.asarray(a, dtype=np.int64))
        return int(arr.size), arr, arr.ctypes.data_as(ctypes.c_void_p)

    nq_, qarr, qp = sel(qrows)
    nk_, karr, kp = sel(kvcols)
    if not want_dq:
        nq_, qarr, qp = 0, np.zeros(1, np.int64), None
        qp = qarr.ctypes.data_as(ctypes.c_void_p)
    if not want_dkv:
        nk_, karr, kp = 0, np.zeros(1, np.int64), None
        kp = karr.ctypes.data_as(ctypes.c_void_p)
    dQ = np.zeros((max(nq_, 1), Hq, D), np.float64)
    dK = np.zeros((max(nk_, 1), Hkv, D), np.float64)
    dV = np.zeros((max(nk_, 1), Hkv, D), np.float64)
    rc = lib.or_attn_bwd(T, Hq, Hkv, D, float(scale), Qd, Kd, Vd, dOd,
                         lab.node_of if T else np.zeros(1, np.int32), lab.parent,
                         nq_, qp, dQ.ctypes.data_as(ctypes.c_void_p) if want_dq else None,
                         nk_, kp, dK.ctypes.data_as(ctypes.c_void_p) if want_dkv else None,
                         dV.ctypes.data_as(ctypes.c_void_p) if want_dkv else None,
                         n_threads or default_threads())
    if rc != OR_OK:
        raise OracleError(f"attn_bwd failed (code {rc})")
    return (dQ[:nq_] if want_dq else None, dK[:nk_] if want_dkv else None, dV[:nk_] if want_dkv else None)
