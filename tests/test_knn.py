"""Queries on a built tree: oracle pins for the K-nearest-nodes definition and
the per-node split dimensions, and host-side argument checks (no GPU)."""
import ctypes

import numpy as np
import pytest

import balanced_tree_build_gb300 as kdt
import oracle
from balanced_tree_build_gb300 import _build
from balanced_tree_build_gb300.inputs import make_points


@pytest.fixture(scope="module")
def o():
    return oracle.get()


def test_knn_hand_example(o):
    # distances from (0, 0): node0 0, node1 9, node2 16, node3 2
    tree = np.array([[0, 0], [3, 0], [0, 4], [1, 1]], np.float32)
    nodes, d2 = o.knn(tree, np.array([[0, 0], [3, 1]], np.float32), 3)
    assert nodes.tolist() == [[0, 3, 1], [1, 3, 0]]
    assert d2.tolist() == [[0, 2, 9], [1, 4, 10]]


def test_knn_ties_by_node_and_short_trees(o):
    tree = np.array([[1, 0], [-1, 0], [0, 1], [0, -1], [5, 5]], np.float32)
    nodes, d2 = o.knn(tree, np.zeros((1, 2), np.float32), 4)
    assert nodes.tolist() == [[0, 1, 2, 3]] and d2.tolist() == [[1, 1, 1, 1]]
    nodes, d2 = o.knn(tree[:2], np.zeros((1, 2), np.float32), 4)
    assert nodes.tolist() == [[0, 1, -1, -1]]
    assert d2[0, :2].tolist() == [1, 1] and np.isinf(d2[0, 2:]).all()


def test_dist2_is_the_stated_float32_sum(o):
    rng = np.random.default_rng(3)
    for k in (1, 3, 8):
        for _ in range(200):
            q = (rng.standard_normal(k) * 10).astype(np.float32)
            p = (rng.standard_normal(k) * 10).astype(np.float32)
            d = np.float32(0)
            for c in range(k):  # left to right, every operation rounded to float32
                t = np.float32(q[c] - p[c])
                d = np.float32(d + np.float32(t * t))
            assert np.float32(o.dist2(q, p)).tobytes() == d.tobytes()


def test_knn_matches_scipy_ckdtree(o):
    from scipy.spatial import cKDTree
    tree = make_points("uniform01", 3000, 3, seed=11)
    queries = make_points("uniform01", 200, 3, seed=12)
    nodes, d2 = o.knn(tree, queries, 5)
    ref_d, ref_i = cKDTree(tree.astype(np.float64)).query(queries.astype(np.float64), k=6)
    for i in range(len(queries)):
        gaps = np.diff(ref_d[i] ** 2)
        if (gaps[:5] > 1e-5).all():  # no near-ties at float32 resolution
            assert nodes[i].tolist() == ref_i[i, :5].tolist()
        assert np.allclose(d2[i], ref_d[i, :5] ** 2, rtol=1e-5, atol=1e-7)


def test_knn_results_sorted_and_consistent(o):
    tree = make_points("dup_heavy", 500, 2, seed=4)
    queries = make_points("dup_heavy", 50, 2, seed=5)
    nodes, d2 = o.knn(tree, queries, 16)
    for i in range(len(queries)):
        pairs = list(zip(d2[i].tolist(), nodes[i].tolist()))
        assert pairs == sorted(pairs)
        for d, u in pairs:
            assert np.float32(o.dist2(queries[i], tree[u])) == np.float32(d)
        # nothing outside the list is strictly better than its last pair
        all_d = np.array([o.dist2(queries[i], tree[u]) for u in range(len(tree))], np.float32)
        worst = pairs[-1]
        better = [(all_d[u], u) for u in range(len(tree)) if (all_d[u], u) < worst]
        assert sorted(better) == pairs[:len(better)] and len(better) == 15


def kd_invariant_holds(tree, dims):
    """Every node's split coordinate bounds its subtrees: left <=, right >=."""
    n = len(tree)
    for u in range(n):
        d = dims[u]
        s = tree[u, d]
        for side, ok in ((2 * u + 1, lambda x: x <= s), (2 * u + 2, lambda x: x >= s)):
            stack = [side]
            while stack:
                v = stack.pop()
                if v >= n:
                    continue
                if not ok(tree[v, d]):
                    return False
                stack += [2 * v + 1, 2 * v + 2]
    return True


@pytest.mark.parametrize("mode", [0, 1])
def test_node_dims_make_the_kd_invariant_hold(o, mode):
    pts = make_points("gaussian", 700, 3, seed=8)
    pts[:, 2] *= 4  # give widest mode a preferred dimension near the root
    perm = o.build_tree(pts, mode)
    tree = oracle.gather_points(pts, perm)
    dims = o.node_dims(tree, mode)
    assert kd_invariant_holds(tree, dims)
    if mode == 0:
        assert dims.tolist() == [o.level(u) % 3 for u in range(700)]
    else:
        # the other rule's dimensions do not fit this tree
        assert not kd_invariant_holds(tree, o.node_dims(tree, 0))


def test_node_dims_hand_example(o):
    # root box x [0, 3], y [0, 4]: y; left of the root y is cut to [0, 0]: x
    tree = np.array([[0, 0], [3, 0], [0, 4], [1, 1]], np.float32)
    assert o.node_dims(tree, 1).tolist() == [1, 0, 1, 0]
    assert o.node_dims(tree, 0).tolist() == [0, 1, 1, 0]


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return kdt.lib()


def test_query_calls_reject_bad_arguments(lib):
    fake = ctypes.c_void_p(0x1000)
    assert lib.kdt_node_dims(None, 10, 3, 0, fake, None) == kdt.EINVAL
    assert lib.kdt_node_dims(fake, 10, 3, 0, None, None) == kdt.EINVAL
    assert lib.kdt_node_dims(fake, 0, 3, 0, fake, None) == kdt.EINVAL
    assert lib.kdt_node_dims(fake, 10, 3, 2, fake, None) == kdt.EINVAL
    assert lib.kdt_knn(None, 10, 3, None, fake, 5, 4, fake, fake, None) == kdt.EINVAL
    assert lib.kdt_knn(fake, 10, 3, None, None, 5, 4, fake, fake, None) == kdt.EINVAL
    assert lib.kdt_knn(fake, 10, 3, None, fake, 5, 0, fake, fake, None) == kdt.EINVAL
    assert lib.kdt_knn(fake, 10, 3, None, fake, 5, 65, fake, fake, None) == kdt.EINVAL
    assert lib.kdt_knn(fake, 10, 3, None, fake, -1, 4, fake, fake, None) == kdt.EINVAL
    assert lib.kdt_knn(fake, 10, 0, None, fake, 5, 4, fake, fake, None) == kdt.EINVAL
