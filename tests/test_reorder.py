"""The points in level order (gather) and the in-place build: oracle pins and
host-side argument checks (no GPU needed)."""
import ctypes

import numpy as np
import pytest

import balanced_tree_build_gb300 as kdt
import oracle
from balanced_tree_build_gb300 import _build
from balanced_tree_build_gb300.inputs import make_points


def test_gather_is_row_by_row_copy():
    pts = make_points("uniform01", 37, 3, seed=5)
    perm = np.random.default_rng(1).permutation(37).astype(np.int32)
    out = oracle.gather_points(pts, perm)
    for node in range(37):  # the definition, one row at a time
        assert out[node].tobytes() == pts[perm[node]].tobytes()


def test_gather_identity_and_reverse():
    pts = make_points("gaussian", 50, 4, seed=2)
    ident = np.arange(50, dtype=np.int32)
    assert oracle.gather_points(pts, ident).tobytes() == pts.tobytes()
    rev = ident[::-1].copy()
    assert oracle.gather_points(pts, rev).tobytes() == pts[::-1].tobytes()


def test_gather_keeps_signed_zero_bits():
    pts = np.array([[-0.0, 1.0], [0.0, -0.0], [2.0, 3.0]], dtype=np.float32)
    out = oracle.gather_points(pts, np.array([1, 2, 0], dtype=np.int32))
    assert out.view(np.uint32).tolist() == [[0, 0x80000000], [0x40000000, 0x40400000], [0x80000000, 0x3F800000]]


def test_gather_rejects_non_permutations():
    pts = make_points("uniform01", 5, 2, seed=1)
    for bad in ([0, 1, 2, 3, 3], [0, 1, 2, 3, 5], [-1, 1, 2, 3, 4], [0, 1, 2]):
        with pytest.raises(ValueError):
            oracle.gather_points(pts, np.array(bad, dtype=np.int32))


def test_level_order_points_of_the_tree():
    # root row = the point of rank ss(lChild(0)) under <_0 (the split point), and the
    # gathered rows of a tree are a rearrangement of the input rows
    pts = make_points("uniform01", 10, 2, seed=7)
    perm = oracle.get().build_tree(pts, 0)
    out = oracle.gather_points(pts, perm)
    assert sorted(map(bytes, out)) == sorted(map(bytes, pts))
    order = sorted(range(10), key=lambda i: (pts[i, 0], pts[i, 1], i))
    # N = 10: L = 4, M = 3, ss(lChild(0)) = 3 + min(3, 4) = 6
    assert out[0].tobytes() == pts[order[6]].tobytes()


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return kdt.lib()


def test_gather_and_inplace_reject_bad_arguments(lib):
    fake = ctypes.c_void_p(0x1000)
    other = ctypes.c_void_p(0x100000)
    assert lib.kdt_gather_points(None, 10, 3, fake, other, None) == kdt.EINVAL
    assert lib.kdt_gather_points(fake, 10, 3, None, other, None) == kdt.EINVAL
    assert lib.kdt_gather_points(fake, 10, 3, fake, None, None) == kdt.EINVAL
    assert lib.kdt_gather_points(fake, 0, 3, fake, other, None) == kdt.EINVAL
    assert lib.kdt_gather_points(fake, 10, 0, fake, other, None) == kdt.EINVAL
    assert lib.kdt_gather_points(fake, 10, 33, fake, other, None) == kdt.EINVAL  # k > KDT_MAX_K
    # out overlapping pts
    assert lib.kdt_gather_points(fake, 10, 3, fake, ctypes.c_void_p(0x1000 + 40), None) == kdt.EINVAL
    assert lib.kdt_gather_points(ctypes.c_void_p(0x1000 + 40), 10, 3, fake, fake, None) == kdt.EINVAL
    need = kdt.workspace_bytes(10, 3, 0)
    assert lib.kdt_build_inplace(None, 10, 3, 0, fake, other, need, None) == kdt.EINVAL
    assert lib.kdt_build_inplace(fake, 10, 3, 0, None, other, need, None) == kdt.EINVAL
    assert lib.kdt_build_inplace(fake, 10, 3, 0, fake, None, need, None) == kdt.EINVAL
    assert lib.kdt_build_inplace(fake, 10, 3, 2, fake, other, need, None) == kdt.EINVAL
    assert lib.kdt_build_inplace(fake, 10, 3, 0, fake, other, need - 1, None) == kdt.ENOMEM
    assert lib.kdt_build_inplace(fake, 10, 3, 0, fake, ctypes.c_void_p(0x100001), need, None) == kdt.EINVAL
