"""CPU oracle for the left-balanced k-d tree build (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The CUDA library never imports it and
shares no code with it.  Every tree routine here is a thin ctypes wrapper
around ``kdt_oracle.c``; see that file's header for the passages each routine
follows (the left-balanced tree, and the balanced median-split tree of
Brown's presort-and-partition builder).  ``gather_points`` (the points in level order) is its definition
written out with numpy indexing.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kdt_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")

OK = 0
EINVAL = -1
ENOMEM = -2
ENONFINITE = -4
EINTERNAL = -6


def library_path(mutant: int = 0) -> str:
    name = "libkdt_oracle.so" if mutant == 0 else f"libkdt_oracle_m{mutant}.so"
    return os.path.join(_BUILD_DIR, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FP contraction).

    ``mutant`` > 0 plants one deliberate mistake (used only by the tests that
    show the pins catch it)."""
    out = library_path(mutant)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(_SRC)):
        return out
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_BUILD_DIR)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", f"-DKDO_MUTANT={int(mutant)}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class Oracle:
    """Typed handle on one compiled oracle (the real one, or a mutant)."""

    def __init__(self, mutant: int = 0):
        self.mutant = mutant
        self.lib = ctypes.CDLL(build(mutant))
        L = self.lib
        i64, i32, f32p = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        L.kdo_level.argtypes = [i64]
        L.kdo_level.restype = i32
        L.kdo_num_levels.argtypes = [i64]
        L.kdo_num_levels.restype = i32
        L.kdo_subtree_count.argtypes = [i64, i64]
        L.kdo_subtree_count.restype = i64
        L.kdo_less.argtypes = [f32p, i32, i32, i64, i64]
        L.kdo_less.restype = i32
        L.kdo_widest_dim.argtypes = [f32p, f32p, i32]
        L.kdo_widest_dim.restype = i32
        L.kdo_build.argtypes = [f32p, i64, i32, i32, f32p]
        L.kdo_build.restype = i32
        L.kdo_verify.argtypes = [f32p, i64, i32, i32, f32p, f32p, i64, i32,
                                 ctypes.POINTER(ctypes.c_int64)]
        L.kdo_verify.restype = i32
        L.kdo_brute_force.argtypes = [f32p, i32, i32, i32, f32p]
        L.kdo_brute_force.restype = i64
        L.kdo_node_dims.argtypes = [f32p, i64, i32, i32, f32p]
        L.kdo_node_dims.restype = i32
        L.kdo_dist2.argtypes = [f32p, f32p, i32]
        L.kdo_dist2.restype = ctypes.c_float
        L.kdo_knn_brute.argtypes = [f32p, i64, i32, f32p, i64, i32, f32p, f32p]
        L.kdo_knn_brute.restype = i32
        L.kdo_balanced_slots.argtypes = [i64]
        L.kdo_balanced_slots.restype = i64
        L.kdo_build_balanced.argtypes = [f32p, i64, i32, f32p, i64]
        L.kdo_build_balanced.restype = i32
        L.kdo_verify_balanced.argtypes = [f32p, i64, i32, f32p, i64, ctypes.POINTER(ctypes.c_int64)]
        L.kdo_verify_balanced.restype = i32
        L.kdo_brute_force_balanced.argtypes = [f32p, i32, i32, f32p]
        L.kdo_brute_force_balanced.restype = i64

    # -- notation ---------------------------------------------------------
    def level(self, i: int) -> int:
        return self.lib.kdo_level(i)

    def num_levels(self, n: int) -> int:
        return self.lib.kdo_num_levels(n)

    def subtree_count(self, n: int, t: int) -> int:
        return self.lib.kdo_subtree_count(n, t)

    # -- order / split rule -----------------------------------------------
    def less(self, pts: np.ndarray, p: int, a: int, b: int) -> bool:
        pts = _points(pts)
        return bool(self.lib.kdo_less(pts.ctypes.data, pts.shape[1], p, a, b))

    def widest_dim(self, lo: np.ndarray, hi: np.ndarray) -> int:
        lo = np.ascontiguousarray(lo, dtype=np.float32)
        hi = np.ascontiguousarray(hi, dtype=np.float32)
        return self.lib.kdo_widest_dim(lo.ctypes.data, hi.ctypes.data, lo.size)

    # -- build / verify -----------------------------------------------------
    def build_tree(self, pts: np.ndarray, mode: int = 0) -> np.ndarray:
        pts = _points(pts)
        n, k = pts.shape
        perm = np.empty(n, dtype=np.int32)
        rc = self.lib.kdo_build(pts.ctypes.data, n, k, mode, perm.ctypes.data)
        if rc != OK:
            raise OracleError(rc)
        return perm

    def verify(self, pts: np.ndarray, perm: np.ndarray, mode: int = 0,
               nodes: np.ndarray | None = None, check_perm: bool = True):
        """Returns (ok, bad_node).  bad_node == -1 flags a non-permutation."""
        pts = _points(pts)
        n, k = pts.shape
        perm = np.ascontiguousarray(perm, dtype=np.int32)
        if perm.shape != (n,):
            raise ValueError("perm must have shape (N,)")
        bad = ctypes.c_int64(-2)
        if nodes is None:
            rc = self.lib.kdo_verify(pts.ctypes.data, n, k, mode, perm.ctypes.data,
                                     None, 0, int(check_perm), ctypes.byref(bad))
        else:
            nodes = np.ascontiguousarray(nodes, dtype=np.int64)
            rc = self.lib.kdo_verify(pts.ctypes.data, n, k, mode, perm.ctypes.data,
                                     nodes.ctypes.data, nodes.size, int(check_perm),
                                     ctypes.byref(bad))
        if rc < 0:
            raise OracleError(rc)
        return rc == 0, int(bad.value)

    # -- queries on a built tree (tree_pts = the points in level order) -------
    def node_dims(self, tree_pts: np.ndarray, mode: int = 0) -> np.ndarray:
        """Split dimension of every node (uint8[N])."""
        tree_pts = _points(tree_pts)
        n, k = tree_pts.shape
        dims = np.empty(n, dtype=np.uint8)
        rc = self.lib.kdo_node_dims(tree_pts.ctypes.data, n, k, mode, dims.ctypes.data)
        if rc != OK:
            raise OracleError(rc)
        return dims

    def dist2(self, q: np.ndarray, p: np.ndarray) -> float:
        q = np.ascontiguousarray(q, dtype=np.float32)
        p = np.ascontiguousarray(p, dtype=np.float32)
        return float(self.lib.kdo_dist2(q.ctypes.data, p.ctypes.data, q.size))

    def knn(self, tree_pts: np.ndarray, queries: np.ndarray, K: int):
        """Brute-force K nearest nodes: (node int32[Q, K], dist2 float32[Q, K])."""
        tree_pts = _points(tree_pts)
        queries = _points(queries)
        n, k = tree_pts.shape
        if queries.shape[1] != k:
            raise ValueError("queries must have k columns")
        qn = queries.shape[0]
        nodes = np.empty((qn, K), dtype=np.int32)
        d2 = np.empty((qn, K), dtype=np.float32)
        rc = self.lib.kdo_knn_brute(tree_pts.ctypes.data, n, k, queries.ctypes.data, qn, K,
                                    nodes.ctypes.data, d2.ctypes.data)
        if rc != OK:
            raise OracleError(rc)
        return nodes, d2

    def brute_force(self, pts: np.ndarray, mode: int = 0):
        """Returns (number of valid orderings, first valid ordering)."""
        pts = _points(pts)
        n, k = pts.shape
        first = np.full(n, -1, dtype=np.int32)
        cnt = self.lib.kdo_brute_force(pts.ctypes.data, n, k, mode, first.ctypes.data)
        if cnt < 0:
            raise OracleError(int(cnt))
        return int(cnt), first


    # -- the balanced (median-split) tree of Brown's builder ----------------
    def balanced_slots(self, n: int) -> int:
        """Heap slots of the balanced tree of n points: 2^numLevels(n) - 1."""
        return int(self.lib.kdo_balanced_slots(n))

    def build_balanced(self, pts: np.ndarray) -> np.ndarray:
        """slots[s] = input index at heap slot s, -1 where a subtree is empty."""
        pts = _points(pts)
        n, k = pts.shape
        slots = np.empty(self.balanced_slots(n), dtype=np.int32)
        rc = self.lib.kdo_build_balanced(pts.ctypes.data, n, k, slots.ctypes.data, slots.size)
        if rc != OK:
            raise OracleError(rc)
        return slots

    def verify_balanced(self, pts: np.ndarray, slots: np.ndarray):
        """Returns (ok, bad_slot): shape, permutation and the k-d condition of
        every node against every ancestor (bad_slot -1: shape or permutation)."""
        pts = _points(pts)
        n, k = pts.shape
        slots = np.ascontiguousarray(slots, dtype=np.int32)
        bad = ctypes.c_int64(-2)
        rc = self.lib.kdo_verify_balanced(pts.ctypes.data, n, k, slots.ctypes.data, slots.size,
                                          ctypes.byref(bad))
        if rc < 0:
            raise OracleError(rc)
        return rc == 0, int(bad.value)

    def brute_force_balanced(self, pts: np.ndarray):
        """Returns (number of valid assignments, first valid slot array)."""
        pts = _points(pts)
        n, k = pts.shape
        first = np.full(self.balanced_slots(n), -1, dtype=np.int32)
        cnt = self.lib.kdo_brute_force_balanced(pts.ctypes.data, n, k, first.ctypes.data)
        if cnt < 0:
            raise OracleError(int(cnt))
        return int(cnt), first


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"oracle returned error code {code}")
        self.code = code


def _points(pts: np.ndarray) -> np.ndarray:
    pts = np.ascontiguousarray(pts, dtype=np.float32)
    if pts.ndim != 2:
        raise ValueError("points must be an (N, k) array")
    return pts


_default: Oracle | None = None


def get() -> Oracle:
    """The (unmutated) oracle, compiled on first use."""
    global _default
    if _default is None:
        _default = Oracle(0)
    return _default


def gather_points(pts: np.ndarray, perm: np.ndarray) -> np.ndarray:
    """The points in level order: row ``node`` of the result is row
    ``perm[node]`` of ``pts``, copied as raw 32-bit words (signed zeros kept).
    "GPU-friendly, Parallel, and (Almost-)In-Place Construction of
    Left-Balanced k-d Trees" (introduction, core idea): the build leaves the
    data array itself in the tree's order.  ``perm`` must be a permutation of
    0..N-1."""
    pts = _points(pts)
    perm = np.asarray(perm)
    n = pts.shape[0]
    if perm.shape != (n,) or not np.issubdtype(perm.dtype, np.integer):
        raise ValueError("perm must be an integer array of shape (N,)")
    if n and (perm.min() < 0 or perm.max() >= n or np.unique(perm).size != n):
        raise ValueError("perm must be a permutation of 0..N-1")
    words = pts.view(np.uint32)
    return np.ascontiguousarray(words[perm.astype(np.int64)]).view(np.float32)
