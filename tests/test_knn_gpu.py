"""Queries on a built tree on the GPU (GPU required): split dimensions and K
nearest nodes, bit-exact against the oracle (node ids and float32 distances)."""
import numpy as np
import pytest
import torch

import balanced_tree_build_gb300 as kdt
import oracle
from balanced_tree_build_gb300.inputs import make_points
from gpu_util import ensure_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def o():
    ensure_library()
    return oracle.get()


def gpu_tree(pts, mode):
    d = torch.from_numpy(pts).cuda()
    perm = kdt.build_inplace(d, mode)
    kdt.check_status()
    return d, perm


@pytest.mark.parametrize("dist,k", [("uniform01", 3), ("gaussian", 2), ("quant1024", 8), ("dup_heavy", 5),
                                    ("signed_zero", 3), ("all_equal", 4), ("uniform01", 32)])
@pytest.mark.parametrize("mode", [0, 1])
def test_node_dims_match_oracle(o, dist, k, mode):
    pts = make_points(dist, 3001, k, seed=k + 17)
    tree, _ = gpu_tree(pts, mode)
    dims = kdt.node_dims(tree, mode)
    kdt.check_status()
    assert np.array_equal(dims.cpu().numpy(), o.node_dims(tree.cpu().numpy(), mode))


def check_knn(o, tree_np, queries_np, K, mode, tree=None, dims=None):
    tree = torch.from_numpy(tree_np).cuda() if tree is None else tree
    q = torch.from_numpy(queries_np).cuda()
    if mode == 1 and dims is None:
        dims = kdt.node_dims(tree, mode)
    nodes, d2 = kdt.knn(tree, q, K, dims=dims if mode == 1 else None)
    kdt.check_status()
    want_n, want_d = o.knn(tree_np, queries_np, K)
    got_n, got_d = nodes.cpu().numpy(), d2.cpu().numpy()
    if not (np.array_equal(got_n, want_n) and np.array_equal(got_d.view(np.uint32), want_d.view(np.uint32))):
        bad = np.nonzero((got_n != want_n).any(axis=1) | (got_d != want_d).any(axis=1))[0]
        raise AssertionError(f"{bad.size} queries differ, first {bad[0]}: gpu {got_n[bad[0]]} {got_d[bad[0]]} "
                             f"oracle {want_n[bad[0]]} {want_d[bad[0]]}")


@pytest.mark.parametrize("dist,k", [("uniform01", 3), ("gaussian", 3), ("dup_heavy", 2), ("signed_zero", 3),
                                    ("all_equal", 3), ("int_grid", 4), ("quant1024", 8),
                                    ("gaussian", 32)])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("K", [1, 4, 16])
def test_knn_matches_oracle(o, dist, k, mode, K):
    pts = make_points(dist, 2500, k, seed=3 * k + K)
    tree, _ = gpu_tree(pts, mode)
    queries = make_points(dist, 300, k, seed=99 + k)
    queries[:20] = tree.cpu().numpy()[::125][:20]  # queries sitting exactly on tree points
    check_knn(o, tree.cpu().numpy(), queries, K, mode, tree=tree)


@pytest.mark.parametrize("n", [1, 2, 3, 7, 64, 65])
def test_knn_small_trees_and_k_beyond_n(o, n):
    pts = make_points("uniform_pm1", n, 3, seed=n)
    tree, _ = gpu_tree(pts, 0)
    check_knn(o, tree.cpu().numpy(), make_points("uniform_pm1", 40, 3, seed=5), 64, 0, tree=tree)


def test_knn_larger_tree(o):
    pts = make_points("mixture64_dup5", 200_000, 3, seed=21)
    tree, _ = gpu_tree(pts, 0)
    queries = make_points("mixture64_dup5", 1000, 3, seed=22)
    check_knn(o, tree.cpu().numpy(), queries, 8, 0, tree=tree)


def test_knn_reports_bad_dims():
    pts = make_points("uniform01", 100, 3, seed=1)
    tree, _ = gpu_tree(pts, 1)
    dims = torch.full((100,), 7, dtype=torch.uint8, device="cuda")
    kdt.knn(tree, tree[:5].clone(), 2, dims=dims)
    assert kdt.status() == kdt.EINVAL
