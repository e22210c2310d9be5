"""The points in level order and the in-place build on the GPU (GPU required):
bit-exact against the oracle's gather of the oracle's tree."""
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


def bits(a) -> np.ndarray:
    a = a.cpu().numpy() if isinstance(a, torch.Tensor) else a
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


@pytest.mark.parametrize("k", [1, 2, 3, 4, 5, 8, 16, 32])
@pytest.mark.parametrize("n", [1, 2, 7, 1000, 4097])
def test_gather_matches_oracle(o, k, n):
    pts = make_points("signed_zero" if k % 2 else "gaussian", n, k, seed=n + k)
    perm = o.build_tree(pts, 0)
    d = torch.from_numpy(pts).cuda()
    out = kdt.gather_points(d, torch.from_numpy(perm).cuda())
    kdt.check_status()
    assert np.array_equal(bits(out), bits(oracle.gather_points(pts, perm)))


@pytest.mark.parametrize("k", [2, 4])
def test_gather_unaligned_rows(o, k):
    # rows of 2 or 4 words starting 4 bytes off a 16-byte boundary take the per-word path
    n = 3001
    pts = make_points("uniform_pm1", n, k, seed=9)
    store = torch.zeros(n * k + 1, dtype=torch.float32, device="cuda")
    store[1:] = torch.from_numpy(pts.reshape(-1)).cuda()
    d = store[1:].view(n, k)
    out_store = torch.zeros(n * k + 1, dtype=torch.float32, device="cuda")
    out = out_store[1:].view(n, k)
    perm = o.build_tree(pts, 1)
    kdt.gather_points(d, torch.from_numpy(perm).cuda(), out=out)
    kdt.check_status()
    assert np.array_equal(bits(out), bits(oracle.gather_points(pts, perm)))


@pytest.mark.parametrize("dist,k,mode", [("uniform01", 3, 0), ("signed_zero", 3, 1), ("dup_heavy", 5, 0),
                                         ("quant1024", 8, 1), ("all_equal", 2, 0)])
@pytest.mark.parametrize("n", [1, 100, 4096, 70001])
def test_build_inplace_matches_oracle(o, dist, k, mode, n):
    pts = make_points(dist, n, k, seed=3 * n + k)
    want_perm = o.build_tree(pts, mode)
    d = torch.from_numpy(pts).cuda()
    perm = kdt.build_inplace(d, mode)
    kdt.check_status()
    assert np.array_equal(perm.cpu().numpy(), want_perm)
    assert np.array_equal(bits(d), bits(oracle.gather_points(pts, want_perm)))


def test_build_inplace_keeps_points_on_error():
    pts = make_points("uniform01", 5000, 3, seed=4)
    pts[1234, 1] = np.nan
    d = torch.from_numpy(pts).cuda()
    kdt.build_inplace(d, 0)
    assert kdt.status() == kdt.ENONFINITE
    assert np.array_equal(bits(d), bits(pts))


def test_gather_reports_bad_permutation():
    pts = make_points("uniform01", 64, 3, seed=4)
    d = torch.from_numpy(pts).cuda()
    perm = torch.arange(64, dtype=torch.int32, device="cuda")
    perm[10] = 64
    out = torch.zeros_like(d)
    kdt.gather_points(d, perm, out=out)
    assert kdt.status() == kdt.EINVAL
    got = out.cpu().numpy()
    assert np.array_equal(bits(got[:10]), bits(pts[:10])) and not got[10].any()


def test_build_inplace_full_size():
    # the largest workload: the rewritten points are the rows the build's
    # permutation names, and the permutation passes the GPU verifier
    w = WORKLOADS["mixture_dup_10m"]
    pts = w.points()
    d = torch.from_numpy(pts).cuda()
    ref = d.clone()
    perm = kdt.build_inplace(d, w.mode)
    kdt.check_status()
    assert kdt.verify_tree(ref, perm, w.mode)
    idx = torch.randint(0, w.n, (100_000,), device="cuda")
    assert torch.equal(d[idx].view(torch.int32), ref[perm[idx].long()].view(torch.int32))
