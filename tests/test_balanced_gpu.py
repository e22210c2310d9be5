"""Parity of the balanced (median-split) tree of Brown's builder with the CPU
oracle (GPU required).

"An Implementation of a Balanced Kd Tree Builder Using GPUs", overview list
and build section: lower median (rank floor((n-1)/2)), split dimension level
mod k, heap-ordered slots with -1 for empty subtrees.  The tree is unique
under the strict super key + index order, so the comparison is bit-exact.
"""
import numpy as np
import pytest
import torch

import balanced_tree_build_gb300 as kdt
import oracle
from balanced_tree_build_gb300.inputs import WORKLOADS, make_points
from gpu_util import ensure_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def o():
    ensure_library()
    return oracle.get()


def gpu_balanced(pts: np.ndarray) -> np.ndarray:
    d = torch.from_numpy(np.ascontiguousarray(pts, dtype=np.float32)).cuda()
    slots = kdt.build_balanced(d)
    kdt.check_status()
    return slots.cpu().numpy()


def assert_parity(o, pts):
    want = o.build_balanced(pts)
    got = gpu_balanced(pts)
    if not np.array_equal(got, want):
        bad = np.nonzero(got != want)[0]
        raise AssertionError(f"{bad.size} slots differ, first at slot {bad[0]}: gpu {got[bad[0]]} "
                             f"oracle {want[bad[0]]} (N={len(pts)}, k={pts.shape[1]})")


SIZES = [1, 2, 3, 4, 5, 7, 8, 9, 15, 16, 17, 31, 32, 33, 100, 255, 256, 257, 1000, 2047, 2048, 4095, 4096,
         4097, 8191, 8192, 8193, 12000, 16385, 40000, 65537]


@pytest.mark.parametrize("n", SIZES)
def test_sizes_uniform(o, n):
    assert_parity(o, make_points("uniform01", n, 3, seed=n))


@pytest.mark.parametrize("dist", ["dup_heavy", "all_equal", "signed_zero", "int_grid", "sorted", "reversed",
                                  "gaussian", "quant1024", "uniform_pm1", "mixture64_dup5"])
@pytest.mark.parametrize("k", [1, 2, 3, 5, 8])
def test_distributions(o, dist, k):
    for n in (37, 777, 5000, 20011):
        assert_parity(o, make_points(dist, n, k, seed=3000 + n + k))


@pytest.mark.parametrize("k", [16, 32])
def test_many_dimensions(o, k):
    for n in (1, 333, 9001):
        assert_parity(o, make_points("uniform01", n, k, seed=n + k))
        assert_parity(o, make_points("dup_heavy", n, k, seed=n + 2 * k))


@pytest.mark.parametrize("n", [100_000, 200_003, 1_000_003])
def test_multi_level_sizes(o, n):
    """Global levels spread over all SMs and one CTA per subtree, then the
    shared-memory finisher."""
    assert_parity(o, make_points("uniform01", n, 3, seed=n))
    assert_parity(o, make_points("dup_heavy", n // 4, 2, seed=n))


@pytest.mark.parametrize("name", ["uniform_1k", "uniform_pm1_1m", "mixture_dup_10m"])
def test_workload_full_size(o, name):
    assert_parity(o, WORKLOADS[name].points())


def test_slots_and_holes():
    ensure_library()
    for n in (1, 2, 3, 6, 10, 1000):
        assert kdt.balanced_slots(n) == 2 ** n.bit_length() - 1
    got = gpu_balanced(make_points("uniform01", 10, 2, seed=0))
    assert got.size == 15 and (got < 0).sum() == 5
    assert np.array_equal(np.sort(got[got >= 0]), np.arange(10))
