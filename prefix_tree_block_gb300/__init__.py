"""prefix_tree_block_gb300 -- prefix-tree attention (forward and backward) for
one NVIDIA GB300, as a C-ABI library (libpt.so, declared in include/pt.h)
with this thin Python binding.

The binding only marshals arguments: it passes raw device pointers and the
current CUDA stream to the library and allocates outputs with PyTorch.  Every
step of the computation runs in the library's CUDA kernels; if libpt.so is
missing the calls raise, there is no other implementation behind them.
Build the library with ``prefix_tree_block_gb300.build.build()``.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

__all__ = [
    "PTError", "BlockMap", "HostStep", "load_library", "build_blockmap_tree", "build_blockmap_seg",
    "build_blockmap_draft",
    "attn_fwd", "attn_bwd", "bwd_workspace_bytes", "sync_status", "launch_count", "LIB_PATH",
    "profile_enable", "profile_read", "profile_reset", "attn_bwd_noalloc", "FoldPlan", "fold_plan",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpt.so")

PT_OK, PT_ERR_INVALID_ARG, PT_ERR_UNSUPPORTED, PT_ERR_CUDA, PT_ERR_TIMEOUT, PT_ERR_NOMEM = range(6)
PT_BF16, PT_F32 = 0, 1
_STATUS_NAMES = {0: "PT_OK", 1: "PT_ERR_INVALID_ARG", 2: "PT_ERR_UNSUPPORTED", 3: "PT_ERR_CUDA",
                 4: "PT_ERR_TIMEOUT", 5: "PT_ERR_NOMEM"}

_lib = None
_lock = threading.Lock()
_alloc_hook = None


def set_output_allocator(fn=None):
    """Route the binding's device output allocations (O, LSE, gradients,
    workspaces, fold outputs) through fn(shape, dtype, device) -> tensor, or
    back to torch.empty with None.  Tests use it to surround every output
    with guard bands."""
    global _alloc_hook
    _alloc_hook = fn


def _empty(shape, dtype, device):
    import torch

    if _alloc_hook is not None:
        return _alloc_hook(tuple(shape), dtype, device)
    return torch.empty(tuple(shape), dtype=dtype, device=device)


class PTError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def load_library(path: Optional[str] = None):
    """Load libpt.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with prefix_tree_block_gb300.build.build()")
        lib = ctypes.CDLL(p)
        vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        pp = ctypes.POINTER(ctypes.c_void_p)
        i32p, i64p = ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)
        sig = {
            "pt_build_blockmap_tree": [vp, i32, vp, vp, i32, i32, i32, vp, pp],
            "pt_build_blockmap_seg": [vp, vp, i32, i32, i32, vp, pp],
            "pt_blockmap_dense": [vp, vp, pp],
            "pt_build_blockmap_draft": [i32, i32, i32, vp, vp, i32, i32, vp, vp, i32, i32, vp, pp],
            "pt_blockmap_info": [vp, i32p, i32p, i32p, i32p, i32p, i64p, i64p],
            "pt_blockmap_export": [vp, vp, vp, vp, vp, vp, vp],
            "pt_blockmap_export_masks": [vp, vp, vp, vp, vp],
            "pt_attn_fwd": [vp, vp, vp, ctypes.c_int, i32, i32, i32, i32, f32, vp, vp, vp, vp],
            "pt_attn_bwd": [vp, vp, vp, vp, vp, vp, ctypes.c_int, i32, i32, i32, i32, f32, vp, vp, vp, vp, vp, sz, vp],
            "pt_sync_status": [vp],
            "pt_debug_wait_timeout": [vp],
            "pt_debug_exp2": [vp, vp, i64, i32, vp],
            "pt_debug_pack_dkdv": [vp, i32, i32, i32, i32, i32, i32, vp, i64, vp, i32p, i32p, i32p],
            "pt_debug_pack_dq": [vp, i32, i32, i32, vp, i64, vp, i32p, i32p, i32p],
            "pt_debug_tree_lists": [vp, i32, vp, vp, i32, i32, i32, vp, i64, vp, i64, i64p],
            "pt_debug_draft_lists": [i32, i32, i32, vp, vp, i32, i32, vp, vp, vp, i64, vp, i64, i64p, i64p],
            "pt_blockmap_prepare_bwd": [vp, i32, i32, i32, vp],
            "pt_attn_bwd_noalloc": [vp, vp, vp, vp, vp, vp, ctypes.c_int, i32, i32, i32, i32, f32, vp, vp, vp, vp,
                                    vp],
            "pt_hoststep_create": [ctypes.c_int, i32, i32, i32, i32, pp],
            "pt_hoststep_run": [vp, vp, vp, vp, vp, f32, vp, vp, vp, vp, vp],
            "pt_hoststep_sync": [vp, vp],
            "pt_hoststep_last_forward": [vp, vp, vp],
            "pt_fold_plan": [vp, i32, vp, vp, i32, i32, vp, pp],
            "pt_foldplan_info": [vp, i32p, i32p, i32p],
            "pt_fold": [vp, vp, i64, vp, vp],
            "pt_unfold": [vp, vp, i64, vp, vp],
            "pt_unfold_grad": [vp, vp, ctypes.c_int, i64, vp, vp],
            "pt_fold_positions": [vp, vp, vp],
            "pt_fold_mismatches": [vp, vp, i64, vp, vp],
            "pt_debug_pool_usage": [i32, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64)],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.pt_blockmap_free.argtypes = [vp]
        lib.pt_blockmap_free.restype = None
        lib.pt_foldplan_free.argtypes = [vp]
        lib.pt_foldplan_free.restype = None
        lib.pt_hoststep_free.argtypes = [vp]
        lib.pt_hoststep_free.restype = None
        lib.pt_bwd_workspace_bytes.argtypes = [i32, i32, i32]
        lib.pt_bwd_workspace_bytes.restype = sz
        lib.pt_last_error.argtypes = []
        lib.pt_last_error.restype = ctypes.c_char_p
        lib.pt_launch_count.argtypes = []
        lib.pt_launch_count.restype = ctypes.c_uint64
        lib.pt_bwd_noalloc_max_scratch_bytes.argtypes = []
        lib.pt_bwd_noalloc_max_scratch_bytes.restype = sz
        lib.pt_debug_drop_listed_tile.argtypes = [i32]
        lib.pt_debug_drop_listed_tile.restype = None
        lib.pt_profile_enable.argtypes = [ctypes.c_int]
        lib.pt_profile_enable.restype = None
        lib.pt_profile_read.argtypes = [ctypes.c_char_p, i64p, ctypes.POINTER(ctypes.c_double)]
        lib.pt_profile_read.restype = ctypes.c_int
        lib.pt_profile_reset.argtypes = []
        lib.pt_profile_reset.restype = None
        _lib = lib
        return lib


def _check(rc: int):
    if rc != PT_OK:
        msg = load_library().pt_last_error()
        raise PTError(rc, msg.decode() if msg else "")


def _stream(stream=None) -> int:
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _ptr(t) -> int:
    return int(t.data_ptr())


class BlockMap:
    """Owner of a device-resident block map built by the library."""

    def __init__(self, handle: int):
        self._h = ctypes.c_void_p(handle)
        self._lib = load_library()
        T, bm_, bn_, nq, nk = (ctypes.c_int32() for _ in range(5))
        _check(self._lib.pt_blockmap_info(self._h, ctypes.byref(T), ctypes.byref(bm_), ctypes.byref(bn_),
                                          ctypes.byref(nq), ctypes.byref(nk), None, None))
        self.T, self.block_m, self.block_n = T.value, bm_.value, bn_.value
        self.nq, self.nk = nq.value, nk.value
        self._counts = None

    def _list_sizes(self):
        # the list sizes reach the host after the build's device work: asked for lazily
        if self._counts is None:
            nnz, nfull = ctypes.c_int64(), ctypes.c_int64()
            _check(self._lib.pt_blockmap_info(self._h, None, None, None, None, None, ctypes.byref(nnz),
                                              ctypes.byref(nfull)))
            self._counts = (nnz.value, nfull.value)
        return self._counts

    @property
    def nnz(self) -> int:
        """Non-empty tiles (waits for the build on the device the first time)."""
        return self._list_sizes()[0]

    @property
    def n_full(self) -> int:
        """Fully kept tiles (waits for the build on the device the first time)."""
        return self._list_sizes()[1]

    @property
    def handle(self):
        return self._h

    def prepare_bwd(self, Hq: int, Hkv: int, D: int, stream=None):
        """Build the work lists attn_bwd_noalloc needs for this head layout."""
        _check(load_library().pt_blockmap_prepare_bwd(self._h, Hq, Hkv, D, ctypes.c_void_p(_stream(stream))))

    def dense(self, stream=None) -> "BlockMap":
        """The same tree with every tile marked partial (no skipping)."""
        out = ctypes.c_void_p()
        _check(self._lib.pt_blockmap_dense(self._h, ctypes.c_void_p(_stream(stream)), ctypes.byref(out)))
        return BlockMap(out.value)

    def export(self) -> dict:
        """Host copies (numpy) of the q-major list and its kv-major transpose."""
        import numpy as np

        n = max(self.nnz, 1)
        q_ptr = np.zeros(self.nq + 1, np.int32)
        k_ptr = np.zeros(self.nk + 1, np.int32)
        kv_idx = np.zeros(n, np.int32)
        q_idx = np.zeros(n, np.int32)
        kind = np.zeros(n, np.uint8)
        kindT = np.zeros(n, np.uint8)
        _check(self._lib.pt_blockmap_export(self._h, q_ptr.ctypes.data, kv_idx.ctypes.data, kind.ctypes.data,
                                            k_ptr.ctypes.data, q_idx.ctypes.data, kindT.ctypes.data))
        e = self.nnz
        return dict(q_ptr=q_ptr, kv_idx=kv_idx[:e], kind=kind[:e], k_ptr=k_ptr, q_idx=q_idx[:e], kindT=kindT[:e],
                    nnz=e, nq=self.nq, nk=self.nk)

    def export_masks(self) -> dict:
        """Host copies (numpy) of the partial tiles' keep bitmasks."""
        import numpy as np

        npart = self.nnz - self.n_full
        pidx = np.zeros(max(self.nnz, 1), np.int32)
        pidxT = np.zeros(max(self.nnz, 1), np.int32)
        rows = np.zeros((max(npart, 1), 128, 4), np.uint32)
        cols = np.zeros((max(npart, 1), 128, 4), np.uint32)
        _check(self._lib.pt_blockmap_export_masks(self._h, pidx.ctypes.data, pidxT.ctypes.data, rows.ctypes.data,
                                                  cols.ctypes.data))
        return dict(pidx=pidx[: self.nnz], pidxT=pidxT[: self.nnz], mask_rows=rows[:npart], mask_cols=cols[:npart])

    def free(self):
        if self._h is not None and self._h.value:
            self._lib.pt_blockmap_free(self._h)
        self._h = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def build_blockmap_tree(node_lengths, path_ptr, path_nodes, block_m: int = 128, block_n: int = 128,
                        stream=None) -> BlockMap:
    """Block map from (node_lengths, CSR sample paths), all host int32 arrays."""
    import numpy as np

    lib = load_library()
    nl = np.ascontiguousarray(np.asarray(node_lengths, dtype=np.int32))
    pp = np.ascontiguousarray(np.asarray(path_ptr, dtype=np.int32))
    pn = np.ascontiguousarray(np.asarray(path_nodes, dtype=np.int32))
    out = ctypes.c_void_p()
    _check(lib.pt_build_blockmap_tree(nl.ctypes.data if nl.size else None, int(nl.size), pp.ctypes.data,
                                      pn.ctypes.data if pn.size else None, int(pp.size - 1), int(block_m),
                                      int(block_n), ctypes.c_void_p(_stream(stream)), ctypes.byref(out)))
    return BlockMap(out.value)


def build_blockmap_draft(ctx_len: int, anchors, block_size: int, block_keep=None, causal: bool = False,
                         window: int = 0, ctx_doc=None, anchor_doc=None, block_m: int = 128, block_n: int = 128,
                         stream=None) -> BlockMap:
    """Block map of the draft-block (DFlash) mask (pt_build_blockmap_draft):
    context [ctx_len] then len(anchors) blocks of block_size tokens; host arrays."""
    import numpy as np

    lib = load_library()
    an = np.ascontiguousarray(np.asarray(anchors, dtype=np.int32))
    keep = None if block_keep is None else np.ascontiguousarray(np.asarray(block_keep, dtype=np.uint8))
    cd = None if ctx_doc is None else np.ascontiguousarray(np.asarray(ctx_doc, dtype=np.int32))
    ad = None if anchor_doc is None else np.ascontiguousarray(np.asarray(anchor_doc, dtype=np.int32))
    ptr = lambda a: (a.ctypes.data if a.size else None) if a is not None else None
    out = ctypes.c_void_p()
    _check(lib.pt_build_blockmap_draft(int(ctx_len), int(an.size), int(block_size), ptr(an), ptr(keep), int(bool(causal)),
                                       int(window), ptr(cd), ptr(ad), int(block_m), int(block_n),
                                       ctypes.c_void_p(_stream(stream)), ctypes.byref(out)))
    return BlockMap(out.value)


def build_blockmap_seg(group_id, suffix_id, block_m: int = 128, block_n: int = 128, stream=None) -> BlockMap:
    """Block map from per-token segment labels (CUDA int32 tensors [T])."""
    import torch

    lib = load_library()
    for t in (group_id, suffix_id):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.int32 and t.is_contiguous()):
            raise TypeError("group_id and suffix_id must be contiguous CUDA int32 tensors")
    if group_id.numel() != suffix_id.numel():
        raise ValueError("group_id and suffix_id differ in length")
    out = ctypes.c_void_p()
    T = int(group_id.numel())
    _check(lib.pt_build_blockmap_seg(_ptr(group_id) if T else None, _ptr(suffix_id) if T else None, T,
                                     int(block_m), int(block_n), ctypes.c_void_p(_stream(stream)),
                                     ctypes.byref(out)))
    return BlockMap(out.value)


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.bfloat16:
        return PT_BF16
    if t.dtype == torch.float32:
        return PT_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _check_tensors(*ts):
    import torch

    dt = ts[0].dtype
    for t in ts:
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous()):
            raise TypeError("tensors must be contiguous CUDA tensors")
        if t.dtype != dt:
            raise TypeError("all tensors must share one dtype")


def attn_fwd(Q, K, V, bm: BlockMap, scale: float = 0.0, O=None, LSE=None, stream=None) -> Tuple:
    """O [T,Hq,D] and LSE [Hq,T] (fp32).  Q [T,Hq,D], K/V [T,Hkv,D]."""
    import torch

    _check_tensors(Q, K, V)
    T, Hq, D = Q.shape
    Hkv = K.shape[1]
    if O is None:
        O = _empty(Q.shape, Q.dtype, Q.device)
    if LSE is None:
        LSE = _empty((Hq, T), torch.float32, Q.device)
    lib = load_library()
    _check(lib.pt_attn_fwd(_ptr(Q), _ptr(K), _ptr(V), _dtype_code(Q), T, Hq, Hkv, D, float(scale), bm.handle,
                           _ptr(O), _ptr(LSE), ctypes.c_void_p(_stream(stream))))
    return O, LSE


def bwd_workspace_bytes(T: int, Hq: int, D: int) -> int:
    return int(load_library().pt_bwd_workspace_bytes(int(T), int(Hq), int(D)))


def attn_bwd(dO, Q, K, V, O, LSE, bm: BlockMap, scale: float = 0.0, dQ=None, dK=None, dV=None, workspace=None,
             stream=None) -> Tuple:
    """dQ [T,Hq,D], dK/dV [T,Hkv,D] from the upstream gradient dO."""
    import torch

    _check_tensors(dO, Q, K, V, O)
    T, Hq, D = Q.shape
    Hkv = K.shape[1]
    dQ = _empty(Q.shape, Q.dtype, Q.device) if dQ is None else dQ
    dK = _empty(K.shape, K.dtype, K.device) if dK is None else dK
    dV = _empty(V.shape, V.dtype, V.device) if dV is None else dV
    need = bwd_workspace_bytes(T, Hq, D)
    if workspace is None:
        workspace = _empty((need,), torch.uint8, Q.device)
    lib = load_library()
    _check(lib.pt_attn_bwd(_ptr(dO), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), _dtype_code(Q), T, Hq, Hkv, D,
                           float(scale), bm.handle, _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(workspace),
                           workspace.numel() * workspace.element_size(), ctypes.c_void_p(_stream(stream))))
    return dQ, dK, dV


def attn_bwd_noalloc(dO, Q, K, V, O, LSE, bm: BlockMap, scale: float = 0.0, dQ=None, dK=None, dV=None,
                     stream=None) -> Tuple:
    """attn_bwd without a workspace: the library's built-in scratch array is
    used instead (for callers that cannot allocate device memory; calls that
    overlap on the GPU race on that array)."""
    import torch

    _check_tensors(dO, Q, K, V, O)
    T, Hq, D = Q.shape
    Hkv = K.shape[1]
    dQ = _empty(Q.shape, Q.dtype, Q.device) if dQ is None else dQ
    dK = _empty(K.shape, K.dtype, K.device) if dK is None else dK
    dV = _empty(V.shape, V.dtype, V.device) if dV is None else dV
    lib = load_library()
    _check(lib.pt_attn_bwd_noalloc(_ptr(dO), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), _dtype_code(Q), T, Hq,
                                   Hkv, D, float(scale), bm.handle, _ptr(dQ), _ptr(dK), _ptr(dV),
                                   ctypes.c_void_p(_stream(stream))))
    return dQ, dK, dV


def sync_status(stream=None):
    """Synchronise and raise PTError if an in-kernel wait timed out."""
    _check(load_library().pt_sync_status(ctypes.c_void_p(_stream(stream))))


def debug_exp2(x, method: int):
    """2^x on the device with the MUFU instruction (method 0) or the kernels'
    FMA-pipe polynomial (method 1); x is a contiguous float32 CUDA tensor."""
    import torch

    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 CUDA tensor")
    y = _empty(x.shape, x.dtype, x.device)
    _check(load_library().pt_debug_exp2(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()), x.numel(),
                                        method, ctypes.c_void_p(_stream(None))))
    return y


def launch_count() -> int:
    return int(load_library().pt_launch_count())


def profile_enable(on: bool = True):
    """Start (or stop) per-kernel CUDA-event timing inside the library."""
    load_library().pt_profile_enable(1 if on else 0)


def profile_read(kernel: str):
    """(launches, total milliseconds) recorded for one kernel name."""
    n, ms = ctypes.c_int64(), ctypes.c_double()
    _check(load_library().pt_profile_read(kernel.encode(), ctypes.byref(n), ctypes.byref(ms)))
    return int(n.value), float(ms.value)


def profile_reset():
    load_library().pt_profile_reset()


class HostStep:
    """Forward and backward from pinned host tensors, double-buffered on the
    device so that consecutive run() calls overlap their copies with the
    kernels (pt_hoststep_*).  Host tensors: Q, dO, dQ [T, Hq, D]; K, V, dK,
    dV [T, Hkv, D], contiguous, of the dtype given at creation."""

    def __init__(self, dtype, T: int, Hq: int, Hkv: int, D: int):
        import torch

        self._lib = load_library()
        self._dt = dtype
        self._code = PT_BF16 if dtype == torch.bfloat16 else PT_F32 if dtype == torch.float32 else None
        if self._code is None:
            raise TypeError("HostStep: dtype must be torch.bfloat16 or torch.float32")
        self.shape = (T, Hq, Hkv, D)
        out = ctypes.c_void_p()
        _check(self._lib.pt_hoststep_create(self._code, T, Hq, Hkv, D, ctypes.byref(out)))
        self._h = out

    def run(self, Q, K, V, dO, bm: BlockMap, dQ, dK, dV, scale: float = 0.0, stream=None):
        """Queue one step; the host outputs are valid after sync() and a
        synchronisation of the stream."""
        T, Hq, Hkv, D = self.shape
        for t, h in ((Q, Hq), (dO, Hq), (dQ, Hq), (K, Hkv), (V, Hkv), (dK, Hkv), (dV, Hkv)):
            if t.is_cuda or t.dtype != self._dt or tuple(t.shape) != (T, h, D) or not t.is_contiguous():
                raise ValueError("HostStep.run: host tensors of the creation dtype and shape expected")
        _check(self._lib.pt_hoststep_run(self._h, _ptr(Q), _ptr(K), _ptr(V), _ptr(dO), float(scale), bm.handle,
                                         _ptr(dQ), _ptr(dK), _ptr(dV), ctypes.c_void_p(_stream(stream))))

    def sync(self, stream=None):
        """Make the stream wait for every download queued so far."""
        _check(self._lib.pt_hoststep_sync(self._h, ctypes.c_void_p(_stream(stream))))

    def last_forward(self):
        """O [T, Hq, D] and LSE [Hq, T] of the most recent run(), as new host
        tensors (waits for that step's kernels)."""
        import torch

        T, Hq, Hkv, D = self.shape
        O = torch.empty((T, Hq, D), dtype=self._dt)
        L = torch.empty((Hq, T), dtype=torch.float32)
        _check(self._lib.pt_hoststep_last_forward(self._h, _ptr(O), _ptr(L)))
        return O, L

    def free(self):
        if self._h is not None and self._h.value:
            self._lib.pt_hoststep_free(self._h)
        self._h = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


class FoldPlan:
    """Shared-prefix fold of rollouts and its inverse (pt_fold_plan and the
    calls after it): the flat layout of the tree (node_lengths, CSR sample
    paths) against n_samples rollout rows of row_len tokens.  Tensors carry
    one row of data per token: flat [T, ...], rollouts [n_samples, row_len, ...]."""

    def __init__(self, node_lengths, path_ptr, path_nodes, row_len: int, stream=None):
        import numpy as np

        self._lib = load_library()
        nl = np.ascontiguousarray(np.asarray(node_lengths, dtype=np.int32))
        pp = np.ascontiguousarray(np.asarray(path_ptr, dtype=np.int32))
        pn = np.ascontiguousarray(np.asarray(path_nodes, dtype=np.int32))
        out = ctypes.c_void_p()
        _check(self._lib.pt_fold_plan(nl.ctypes.data if nl.size else None, int(nl.size), pp.ctypes.data,
                                      pn.ctypes.data if pn.size else None, int(pp.size - 1), int(row_len),
                                      ctypes.c_void_p(_stream(stream)), ctypes.byref(out)))
        self._h = out
        T, S, L = (ctypes.c_int32() for _ in range(3))
        _check(self._lib.pt_foldplan_info(self._h, ctypes.byref(T), ctypes.byref(S), ctypes.byref(L)))
        self.T, self.n_samples, self.row_len = T.value, S.value, L.value

    @staticmethod
    def _row_bytes(t, lead: int) -> int:
        """Bytes of one token's row: the trailing dimensions (valid for empty leading ones)."""
        n = t.element_size()
        for d in t.shape[lead:]:
            n *= d
        return n

    def _need(self, t, shape, name):
        if not t.is_cuda or not t.is_contiguous() or tuple(t.shape[:len(shape)]) != shape:
            raise ValueError(f"{name} must be a contiguous CUDA tensor of leading shape {shape}")

    def fold(self, roll, out=None, stream=None):
        """flat[t] = roll[first sample holding t][its position]."""
        import torch

        self._need(roll, (self.n_samples, self.row_len), "roll")
        rb = self._row_bytes(roll, 2)
        out = _empty((self.T,) + tuple(roll.shape[2:]), roll.dtype, roll.device) if out is None else out
        _check(self._lib.pt_fold(self._h, _ptr(roll), rb, _ptr(out), ctypes.c_void_p(_stream(stream))))
        return out

    def unfold(self, flat, out=None, stream=None):
        """roll[s][j] = flat[token at position j of sample s]; padding zero."""
        import torch

        self._need(flat, (self.T,), "flat")
        rb = self._row_bytes(flat, 1)
        out = _empty((self.n_samples, self.row_len) + tuple(flat.shape[1:]), flat.dtype, flat.device) \
            if out is None else out
        _check(self._lib.pt_unfold(self._h, _ptr(flat), rb, _ptr(out), ctypes.c_void_p(_stream(stream))))
        return out

    def unfold_grad(self, droll, out=None, stream=None):
        """dflat[t] = sum of droll over every copy of t (fp32 sums, rounded once)."""
        import torch

        self._need(droll, (self.n_samples, self.row_len), "droll")
        width = 1
        for d in droll.shape[2:]:
            width *= d
        out = _empty((self.T,) + tuple(droll.shape[2:]), droll.dtype, droll.device) if out is None else out
        _check(self._lib.pt_unfold_grad(self._h, _ptr(droll), _dtype_code(droll), width, _ptr(out),
                                        ctypes.c_void_p(_stream(stream))))
        return out

    def positions(self, device=None, stream=None):
        """Position ids of the flat tokens (int64 [T])."""
        import torch

        out = _empty((self.T,), torch.int64, device or torch.device("cuda"))
        _check(self._lib.pt_fold_positions(self._h, _ptr(out), ctypes.c_void_p(_stream(stream))))
        return out

    def mismatches(self, roll, stream=None) -> int:
        """Rollout entries whose bytes differ from the entry the fold keeps (synchronises)."""
        import torch

        self._need(roll, (self.n_samples, self.row_len), "roll")
        cnt = _empty((1,), torch.int64, roll.device)
        _check(self._lib.pt_fold_mismatches(self._h, _ptr(roll), self._row_bytes(roll, 2), _ptr(cnt),
                                            ctypes.c_void_p(_stream(stream))))
        return int(cnt.item())

    def free(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.pt_foldplan_free(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def fold_plan(node_lengths, path_ptr, path_nodes, row_len: int, stream=None) -> FoldPlan:
    """Plan of the shared-prefix fold for a tree and a rollout row length."""
    return FoldPlan(node_lengths, path_ptr, path_nodes, row_len, stream)
