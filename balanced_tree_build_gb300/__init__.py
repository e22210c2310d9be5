"""GB300-native builder for left-balanced, complete, level-order k-d trees.

Thin Python binding over the C ABI in ``include/kdtree_build.h``: the
functions here only check and marshal arguments (torch tensors give device
memory and the current CUDA stream); every step of the build runs in the
library's CUDA kernels.  There is no CPU fallback: if the compiled library is
missing, the calls raise.

    import torch, balanced_tree_build_gb300 as kdt
    pts = torch.rand(1_000_000, 3, device="cuda")
    perm = kdt.build_tree(pts)          # int32 [N]: perm[node] = input index
    assert kdt.verify_tree(pts, perm)
"""
from __future__ import annotations

import ctypes
import os
import re

SPLIT_ROUND_ROBIN = 0
SPLIT_WIDEST = 1

OK = 0
EINVAL = -1
ENOMEM = -2
ECUDA = -3
ENONFINITE = -4
ETIMEOUT = -5
EINTERNAL = -6

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libkdtree_gb300.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "kdtree_build.h")

_lib = None


class KdtError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        msg = _error_string(code)
        super().__init__(f"{what}: {msg} ({code})" if what else f"{msg} ({code})")


class _KernelStat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", ctypes.c_int64),
                ("total_ms", ctypes.c_double), ("bytes_alg", ctypes.c_double), ("kernels", ctypes.c_int64)]


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"CUDA library not built ({LIB_PATH} missing); run "
            "`python -m balanced_tree_build_gb300._build` first")
    L = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    L.kdt_workspace_size.argtypes = [i64, i32, i32, ctypes.POINTER(sz)]
    L.kdt_host_workspace_size.argtypes = [i64, i32, i32, ctypes.POINTER(sz)]
    L.kdt_build.argtypes = [vp, i64, i32, i32, vp, vp]
    L.kdt_build_ws.argtypes = [vp, i64, i32, i32, vp, vp, sz, vp]
    L.kdt_build_host.argtypes = [vp, i64, i32, i32, vp, vp, sz, vp]
    L.kdt_verify.argtypes = [vp, i64, i32, i32, vp, vp]
    L.kdt_gather_points.argtypes = [vp, i64, i32, vp, vp, vp]
    L.kdt_build_inplace.argtypes = [vp, i64, i32, i32, vp, vp, sz, vp]
    L.kdt_node_dims.argtypes = [vp, i64, i32, i32, vp, vp]
    L.kdt_knn.argtypes = [vp, i64, i32, vp, vp, i64, i32, vp, vp, vp]
    L.kdt_balanced_slots.argtypes = [i64, ctypes.POINTER(i64)]
    L.kdt_balanced_workspace_size.argtypes = [i64, i32, ctypes.POINTER(sz)]
    L.kdt_build_balanced.argtypes = [vp, i64, i32, vp, vp, sz, vp]
    L.kdt_status.argtypes = [vp]
    L.kdt_error_string.argtypes = [i32]
    L.kdt_error_string.restype = ctypes.c_char_p
    L.kdt_profile_enable.argtypes = [i32]
    L.kdt_profile_read.argtypes = [ctypes.POINTER(_KernelStat), i32]
    for name in ("kdt_workspace_size", "kdt_host_workspace_size", "kdt_build", "kdt_build_ws",
                 "kdt_build_host", "kdt_verify", "kdt_gather_points", "kdt_build_inplace", "kdt_node_dims",
                 "kdt_knn", "kdt_status", "kdt_balanced_slots", "kdt_balanced_workspace_size",
                 "kdt_build_balanced",
                 "kdt_profile_enable",
                 "kdt_profile_reset", "kdt_profile_read"):
        getattr(L, name).restype = i32
    _lib = L
    return L


def lib():
    """The loaded ctypes library (raises if it was not built)."""
    return _load()


def header_symbols() -> list[str]:
    """Names of the functions declared in include/kdtree_build.h."""
    with open(HEADER_PATH) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(kdt_\w+)\s*\(", text, re.M)))


def _error_string(code: int) -> str:
    try:
        return _load().kdt_error_string(code).decode()
    except Exception:  # library missing: still produce a message
        return {0: "ok", -1: "invalid argument", -2: "out of memory", -3: "CUDA error",
                -4: "non-finite coordinate", -5: "timeout", -6: "internal error"}.get(code, "error")


def _check(rc: int, what: str) -> int:
    if rc < 0:
        raise KdtError(rc, what)
    return rc


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check_points(points):
    import torch
    if not isinstance(points, torch.Tensor):
        raise TypeError("points must be a torch.Tensor")
    if not points.is_cuda:
        raise ValueError("points must be a CUDA tensor (use build_tree_host for host data)")
    if points.dtype != torch.float32 or points.dim() != 2 or not points.is_contiguous():
        raise ValueError("points must be a contiguous float32 tensor of shape (N, k)")
    return points.shape[0], points.shape[1]


def workspace_bytes(n: int, k: int, mode: int = SPLIT_ROUND_ROBIN) -> int:
    out = ctypes.c_size_t(0)
    _check(_load().kdt_workspace_size(n, k, mode, ctypes.byref(out)), "kdt_workspace_size")
    return int(out.value)


def host_workspace_bytes(n: int, k: int, mode: int = SPLIT_ROUND_ROBIN) -> int:
    out = ctypes.c_size_t(0)
    _check(_load().kdt_host_workspace_size(n, k, mode, ctypes.byref(out)), "kdt_host_workspace_size")
    return int(out.value)


def alloc_workspace(n: int, k: int, mode: int = SPLIT_ROUND_ROBIN, device=None, host: bool = False):
    """A device byte tensor big enough for kdt_build_ws (or kdt_build_host)."""
    import torch
    nbytes = host_workspace_bytes(n, k, mode) if host else workspace_bytes(n, k, mode)
    return torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")


def build_tree(points, mode: int = SPLIT_ROUND_ROBIN, out=None, workspace=None, stream=None):
    """Builds the tree of ``points`` (CUDA float32 [N, k]) and returns int32
    [N] with perm[node] = input index.  Stream-ordered on ``stream`` (default:
    torch's current stream).  With ``workspace`` (from alloc_workspace) the
    call allocates nothing; otherwise the library allocates stream-ordered."""
    import torch
    n, k = _check_points(points)
    if out is None:
        out = torch.empty(n, dtype=torch.int32, device=points.device)
    elif out.dtype != torch.int32 or out.shape != (n,) or not out.is_cuda or not out.is_contiguous():
        raise ValueError("out must be a contiguous CUDA int32 tensor of shape (N,)")
    L = _load()
    s = _stream_ptr(stream)
    if workspace is None:
        rc = L.kdt_build(ctypes.c_void_p(points.data_ptr()), n, k, mode,
                         ctypes.c_void_p(out.data_ptr()), s)
    else:
        rc = L.kdt_build_ws(ctypes.c_void_p(points.data_ptr()), n, k, mode,
                            ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(workspace.data_ptr()),
                            workspace.numel() * workspace.element_size(), s)
    _check(rc, "kdt_build")
    return out


def build_tree_host(points, mode: int = SPLIT_ROUND_ROBIN, out=None, workspace=None, stream=None):
    """Host-buffer build: ``points`` is a host float32 [N, k] array (numpy or
    CPU tensor; pinned memory copies asynchronously), the result a host int32
    array.  Synchronous."""
    import numpy as np
    import torch
    if isinstance(points, np.ndarray):
        pts = np.ascontiguousarray(points, dtype=np.float32)
        ptr, n, k = pts.ctypes.data, pts.shape[0], pts.shape[1]
        keep = pts
    else:
        if points.is_cuda or points.dtype != torch.float32 or points.dim() != 2 or not points.is_contiguous():
            raise ValueError("points must be a contiguous host float32 (N, k) array")
        ptr, n, k = points.data_ptr(), points.shape[0], points.shape[1]
        keep = points
    if out is None:
        out = np.empty(n, dtype=np.int32)
    optr = out.ctypes.data if isinstance(out, np.ndarray) else out.data_ptr()
    if workspace is None:
        workspace = alloc_workspace(n, k, mode, host=True)
    rc = _load().kdt_build_host(ctypes.c_void_p(ptr), n, k, mode, ctypes.c_void_p(optr),
                                ctypes.c_void_p(workspace.data_ptr()),
                                workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    del keep
    _check(rc, "kdt_build_host")
    return out


def balanced_slots(n: int) -> int:
    """Heap slots of the balanced (median-split) tree of n points."""
    out = ctypes.c_int64(0)
    _check(_load().kdt_balanced_slots(n, ctypes.byref(out)), "kdt_balanced_slots")
    return int(out.value)


def balanced_workspace_bytes(n: int, k: int) -> int:
    out = ctypes.c_size_t(0)
    _check(_load().kdt_balanced_workspace_size(n, k, ctypes.byref(out)), "kdt_balanced_workspace_size")
    return int(out.value)


def build_balanced(points, out=None, workspace=None, stream=None):
    """Builds the balanced tree of Brown's builder (lower median, split
    dimension level mod k) over ``points`` (CUDA float32 [N, k]); returns int32
    [balanced_slots(N)] in heap order, -1 in the slots of empty subtrees.
    Stream-ordered."""
    import torch
    n, k = _check_points(points)
    slots = balanced_slots(n)
    if out is None:
        out = torch.empty(slots, dtype=torch.int32, device=points.device)
    elif out.dtype != torch.int32 or out.shape != (slots,) or not out.is_cuda or not out.is_contiguous():
        raise ValueError("out must be a contiguous CUDA int32 tensor of shape (balanced_slots(N),)")
    if workspace is None:
        workspace = torch.empty(balanced_workspace_bytes(n, k), dtype=torch.uint8, device=points.device)
    rc = _load().kdt_build_balanced(ctypes.c_void_p(points.data_ptr()), n, k, ctypes.c_void_p(out.data_ptr()),
                                    ctypes.c_void_p(workspace.data_ptr()),
                                    workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check(rc, "kdt_build_balanced")
    return out


def verify_tree(points, perm, mode: int = SPLIT_ROUND_ROBIN, stream=None) -> bool:
    """True iff ``perm`` is the tree of ``points`` (every node against every
    ancestor, plus the permutation check).  Synchronous."""
    import torch
    n, k = _check_points(points)
    if perm.dtype != torch.int32 or perm.shape != (n,) or not perm.is_cuda or not perm.is_contiguous():
        raise ValueError("perm must be a contiguous CUDA int32 tensor of shape (N,)")
    rc = _load().kdt_verify(ctypes.c_void_p(points.data_ptr()), n, k, mode,
                            ctypes.c_void_p(perm.data_ptr()), _stream_ptr(stream))
    _check(rc, "kdt_verify")
    return rc == 0


def gather_points(points, perm, out=None, stream=None):
    """The points in level order: out[node] = points[perm[node]] (CUDA float32
    [N, k], bit-exact).  ``out`` must not overlap ``points``.  Stream-ordered;
    a bad ``perm`` entry shows up in status()."""
    import torch
    n, k = _check_points(points)
    if perm.dtype != torch.int32 or perm.shape != (n,) or not perm.is_cuda or not perm.is_contiguous():
        raise ValueError("perm must be a contiguous CUDA int32 tensor of shape (N,)")
    if out is None:
        out = torch.empty_like(points)
    elif out.dtype != torch.float32 or out.shape != points.shape or not out.is_cuda or not out.is_contiguous():
        raise ValueError("out must be a contiguous CUDA float32 tensor shaped like points")
    rc = _load().kdt_gather_points(ctypes.c_void_p(points.data_ptr()), n, k, ctypes.c_void_p(perm.data_ptr()),
                                   ctypes.c_void_p(out.data_ptr()), _stream_ptr(stream))
    _check(rc, "kdt_gather_points")
    return out


def build_inplace(points, mode: int = SPLIT_ROUND_ROBIN, perm=None, workspace=None, stream=None):
    """Builds the tree of ``points`` (CUDA float32 [N, k]) and rewrites
    ``points`` in level order (row node = the point stored at node); returns
    the int32 permutation.  ``workspace`` (from alloc_workspace) is the only
    temporary; one is allocated if omitted.  Stream-ordered."""
    import torch
    n, k = _check_points(points)
    if perm is None:
        perm = torch.empty(n, dtype=torch.int32, device=points.device)
    elif perm.dtype != torch.int32 or perm.shape != (n,) or not perm.is_cuda or not perm.is_contiguous():
        raise ValueError("perm must be a contiguous CUDA int32 tensor of shape (N,)")
    if workspace is None:
        workspace = alloc_workspace(n, k, mode, device=points.device)
    rc = _load().kdt_build_inplace(ctypes.c_void_p(points.data_ptr()), n, k, mode, ctypes.c_void_p(perm.data_ptr()),
                                   ctypes.c_void_p(workspace.data_ptr()),
                                   workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check(rc, "kdt_build_inplace")
    return perm


def node_dims(tree_points, mode: int = SPLIT_ROUND_ROBIN, out=None, stream=None):
    """Split dimension of every node (CUDA uint8 [N]) of the tree whose points
    in level order are ``tree_points``.  Stream-ordered."""
    import torch
    n, k = _check_points(tree_points)
    if out is None:
        out = torch.empty(n, dtype=torch.uint8, device=tree_points.device)
    elif out.dtype != torch.uint8 or out.shape != (n,) or not out.is_cuda or not out.is_contiguous():
        raise ValueError("out must be a contiguous CUDA uint8 tensor of shape (N,)")
    rc = _load().kdt_node_dims(ctypes.c_void_p(tree_points.data_ptr()), n, k, mode,
                               ctypes.c_void_p(out.data_ptr()), _stream_ptr(stream))
    _check(rc, "kdt_node_dims")
    return out


def knn(tree_points, queries, K: int, dims=None, out_nodes=None, out_dist2=None, stream=None):
    """The K nearest nodes of each query: (int32 [Q, K] node ids, float32
    [Q, K] squared distances), ascending by (dist2, node).  ``dims``: the
    tree's split dimensions (node_dims); None means round-robin.
    Stream-ordered."""
    import torch
    n, k = _check_points(tree_points)
    qn, qk = _check_points(queries)
    if qk != k:
        raise ValueError("queries must have the tree's k columns")
    if out_nodes is None:
        out_nodes = torch.empty((qn, K), dtype=torch.int32, device=queries.device)
    if out_dist2 is None:
        out_dist2 = torch.empty((qn, K), dtype=torch.float32, device=queries.device)
    if dims is not None and (dims.dtype != torch.uint8 or dims.shape != (n,) or not dims.is_cuda):
        raise ValueError("dims must be a CUDA uint8 tensor of shape (N,)")
    rc = _load().kdt_knn(ctypes.c_void_p(tree_points.data_ptr()), n, k,
                         ctypes.c_void_p(dims.data_ptr()) if dims is not None else None,
                         ctypes.c_void_p(queries.data_ptr()), qn, K, ctypes.c_void_p(out_nodes.data_ptr()),
                         ctypes.c_void_p(out_dist2.data_ptr()), _stream_ptr(stream))
    _check(rc, "kdt_knn")
    return out_nodes, out_dist2


def status(stream=None) -> int:
    """Synchronises, then returns and clears the device status word."""
    return int(_load().kdt_status(_stream_ptr(stream)))


def check_status(stream=None) -> None:
    rc = status(stream)
    if rc != OK:
        raise KdtError(rc, "device status")


def profile_enable(on: bool = True) -> None:
    _load().kdt_profile_enable(1 if on else 0)


def profile_reset() -> None:
    _load().kdt_profile_reset()


def profile_read() -> list[dict]:
    L = _load()
    buf = (_KernelStat * 64)()
    n = L.kdt_profile_read(buf, 64)
    return [{"name": buf[i].name.decode(), "launches": int(buf[i].launches),
             "total_ms": float(buf[i].total_ms), "bytes_alg": float(buf[i].bytes_alg),
             "kernels": int(buf[i].kernels)}
            for i in range(min(n, 64))]
