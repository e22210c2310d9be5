"""Parity of the CUDA build with the CPU oracle (GPU required).

The tree is unique under the strict split order, so the comparison is
bit-exact: the permutation from the CUDA library must equal the oracle's,
element by element.  At the largest size the oracle's recursive build is too
slow, so that case is checked by the oracle's verifier (every node against
every ancestor plus the permutation check), which by uniqueness is equivalent.
"""
import numpy as np
import pytest
import torch

import balanced_tree_build_gb300 as kdt
import oracle
import _pins
from balanced_tree_build_gb300.inputs import WORKLOADS, make_points
from gpu_util import ensure_library, gpu_build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def o():
    ensure_library()
    return oracle.get()


def assert_parity(o, pts, mode, **kw):
    want = o.build_tree(pts, mode)
    got = gpu_build(pts, mode, **kw)
    if not np.array_equal(got, want):
        bad = np.nonzero(got != want)[0]
        raise AssertionError(f"{bad.size} nodes differ, first at node {bad[0]}: "
                             f"gpu {got[bad[0]]} oracle {want[bad[0]]} (N={len(pts)}, mode={mode})")


def test_worked_example(o):
    pts, perm, _ = _pins.load_worked_example()
    assert np.array_equal(gpu_build(pts, 0), perm)
    assert np.array_equal(gpu_build(pts, 1), o.build_tree(pts, 1))


SMALL_N = [1, 2, 3, 4, 5, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 64, 65, 100, 255, 256, 257, 258,
           511, 512, 513, 1000, 2047, 4095, 4096, 4097]


@pytest.mark.parametrize("n", SMALL_N)
@pytest.mark.parametrize("mode", [0, 1])
def test_small_sizes_uniform(o, n, mode):
    assert_parity(o, make_points("uniform01", n, 3, seed=n), mode)


@pytest.mark.parametrize("dist", ["dup_heavy", "all_equal", "signed_zero", "int_grid", "sorted",
                                  "reversed", "gaussian", "quant1024", "uniform_pm1"])
@pytest.mark.parametrize("k", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("mode", [0, 1])
def test_distributions(o, dist, k, mode):
    for n in (37, 777, 5000):
        assert_parity(o, make_points(dist, n, k, seed=1000 + n + k), mode)


@pytest.mark.parametrize("n", [8191, 8192, 8193, 12000, 16383, 16384, 16385, 40000, 65537, 200003])
@pytest.mark.parametrize("k,mode", [(3, 0), (3, 1), (8, 1), (1, 0), (2, 0)])
def test_across_tile_boundaries(o, n, k, mode):
    """Sizes that put the switch from the per-level kernel to the shared-memory
    finisher at different levels, with ragged last levels."""
    assert_parity(o, make_points("uniform01", n, k, seed=n * 7 + k), mode)


@pytest.mark.parametrize("n", [40000, 200003])
@pytest.mark.parametrize("k", [4, 5, 6, 7, 8, 16])
@pytest.mark.parametrize("dist", ["uniform01", "dup_heavy"])
def test_round_robin_many_dims_multi_level(o, n, k, dist):
    """Round-robin builds whose global levels run on the whole GPU with the
    next level's histogram fused into the partition: the next split
    coordinate takes every value 0..k-1, including those past the first
    four (held apart from the input index in the partition tile)."""
    assert_parity(o, make_points(dist, n, k, seed=n + 31 * k), 0)


@pytest.mark.parametrize("k", [17, 24, 31, 32])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("dist", ["uniform01", "dup_heavy", "quant1024"])
def test_many_dimensions_up_to_the_limit(o, k, mode, dist):
    """k up to KDT_MAX_K = 32: small tiles (the finisher's shared memory holds
    k key columns), every coordinate split on, and round-robin masks that wrap
    past bit 31."""
    for n in (1, 333, 9_001, 70_003):
        assert_parity(o, make_points(dist, n, k, seed=n + 97 * k + mode), mode)


@pytest.mark.parametrize("dist", ["all_equal", "dup_heavy", "quant1024", "signed_zero"])
def test_heavy_ties_multi_level(o, dist):
    assert_parity(o, make_points(dist, 150_000, 3, seed=5), 0)
    assert_parity(o, make_points(dist, 60_000, 4, seed=6), 1)


def test_allocating_entry_point_matches(o):
    pts = make_points("mixture64_dup5", 50_000, 3, seed=9)
    assert np.array_equal(gpu_build(pts, 0, workspace=False), o.build_tree(pts, 0))


def test_host_buffer_entry_point(o):
    pts = make_points("gaussian", 70_001, 3, seed=10)
    got = kdt.build_tree_host(pts, 0)
    assert np.array_equal(got, o.build_tree(pts, 0))
    pinned = torch.from_numpy(pts).pin_memory()
    got2 = kdt.build_tree_host(pinned, 0)
    assert np.array_equal(got2, got)


@pytest.mark.parametrize("name", ["uniform_1k", "uniform_pm1_1m", "quant1024_k8_4m", "mixture_dup_10m"])
def test_workload_full_size(o, name):
    w = WORKLOADS[name]
    assert_parity(o, w.points(), w.mode)


def test_largest_workload_by_verifier(o):
    """The 100M-point build in the bench's launch configuration (caller
    workspace, one stream), checked by the GPU verifier and by the oracle's
    verifier on every node."""
    w = WORKLOADS["uniform_100m"]
    pts = w.points()
    perm = gpu_build(pts, w.mode)
    assert np.array_equal(np.sort(perm), np.arange(w.n, dtype=np.int32))
    d = torch.from_numpy(pts).cuda()
    assert kdt.verify_tree(d, torch.from_numpy(perm).cuda(), w.mode)
    ok, bad = o.verify(pts, perm, w.mode, check_perm=False)
    assert ok, f"node {bad} violates the tree conditions"


def test_gpu_verifier_rejects_corruption(o):
    ensure_library()
    pts = make_points("dup_heavy", 20_000, 3, seed=12)
    d = torch.from_numpy(pts).cuda()
    for mode in (0, 1):
        perm = torch.from_numpy(o.build_tree(pts, mode)).cuda()
        assert kdt.verify_tree(d, perm, mode)
        bad = perm.clone()
        bad[[10, 9000]] = bad[[9000, 10]]
        assert not kdt.verify_tree(d, bad, mode)
        dup = perm.clone()
        dup[3] = dup[4]
        assert not kdt.verify_tree(d, dup, mode)
        oob = perm.clone()
        oob[7] = 20_000
        assert not kdt.verify_tree(d, oob, mode)


def test_non_finite_input_reports_status():
    ensure_library()
    pts = make_points("uniform01", 10_000, 3, seed=13)
    pts[1234, 1] = np.nan
    d = torch.from_numpy(pts).cuda()
    kdt.build_tree(d, 0)
    assert kdt.status() == kdt.ENONFINITE
    assert kdt.status() == kdt.OK  # cleared by the read
    pts[1234, 1] = np.inf
    with pytest.raises(kdt.KdtError) as e:
        kdt.build_tree_host(pts, 0)
    assert e.value.code == kdt.ENONFINITE
    kdt.status()
    with pytest.raises(kdt.KdtError):
        kdt.verify_tree(torch.from_numpy(pts).cuda(), torch.zeros(10_000, dtype=torch.int32).cuda(), 0)
