"""kdt_build_static: the build entry point that allocates nothing (GPU).

Callers that cannot allocate device memory where they build a tree (a plugin
whose host application owns all device memory, a latency-critical loop where
an allocation could stall or fail) use kdt_build_static, which takes its
scratch from one fixed array that the library reserves on each device.  These
tests call it through the C ABI twice in a row and compare its output with
the CPU oracle and with the regular entry point kdt_build_ws (exact equality:
the tree is unique, so the permutations must match element for element).

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import balanced_tree_build_gb300 as kdt
import oracle
from balanced_tree_build_gb300.inputs import make_points
from gpu_util import ensure_library

pytestmark = pytest.mark.gpu

STATIC_BYTES = 32 * 1024 * 1024  # KDT_STATIC_SCRATCH_BYTES in include/kdtree_build.h


def _static_fn():
    ensure_library()
    fn = kdt.lib().kdt_build_static
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                   ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _build_static(fn, d_pts, mode):
    n, k = d_pts.shape
    out = torch.full((n,), -1, dtype=torch.int32, device=d_pts.device)
    s = torch.cuda.current_stream()
    rc = fn(ctypes.c_void_p(d_pts.data_ptr()), n, k, mode, ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(s.cuda_stream))
    assert rc == kdt.OK, kdt.KdtError(rc, "kdt_build_static")
    torch.cuda.synchronize()
    assert kdt.status() == kdt.OK
    return out.cpu().numpy()


def _build_ws(d_pts, mode):
    n, k = d_pts.shape
    ws = kdt.alloc_workspace(n, k, mode)
    out = kdt.build_tree(d_pts, mode, workspace=ws)
    torch.cuda.synchronize()
    assert kdt.status() == kdt.OK
    return out.cpu().numpy()


def test_header_states_the_limit():
    with open(kdt.HEADER_PATH) as f:
        text = f.read()
    assert "#define KDT_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)" in text
    assert "kdt_build_static" in kdt.header_symbols()


@pytest.mark.parametrize("dist,n,k,mode", [
    ("uniform01", 300_000, 3, 0),
    ("mixture64_dup5", 123_457, 3, 0),
    ("quant1024", 40_000, 8, 1),
    ("dup_heavy", 9_000, 2, 1),
])
def test_matches_regular_entry_point_twice(dist, n, k, mode):
    fn = _static_fn()
    assert kdt.workspace_bytes(n, k, mode) <= STATIC_BYTES
    a = torch.from_numpy(make_points(dist, n, k, seed=41)).cuda()
    b = torch.from_numpy(make_points(dist, n, k, seed=42)).cuda()
    first = _build_static(fn, a, mode)
    second = _build_static(fn, b, mode)  # reuses the array left dirty by the first call
    o = oracle.get()
    assert np.array_equal(first, o.build_tree(a.cpu().numpy(), mode))
    assert np.array_equal(second, o.build_tree(b.cpu().numpy(), mode))
    assert np.array_equal(first, _build_ws(a, mode))
    assert np.array_equal(second, _build_ws(b, mode))


def test_smaller_build_after_larger_one():
    fn = _static_fn()
    big = torch.from_numpy(make_points("uniform01", 400_000, 3, seed=7)).cuda()
    small = torch.from_numpy(make_points("gaussian", 777, 3, seed=8)).cuda()
    _build_static(fn, big, 0)
    got = _build_static(fn, small, 0)
    assert np.array_equal(got, oracle.get().build_tree(small.cpu().numpy(), 0))
    assert np.array_equal(got, _build_ws(small, 0))


def test_rejects_builds_that_do_not_fit():
    fn = _static_fn()
    n = 2_000_000
    assert kdt.workspace_bytes(n, 3, 0) > STATIC_BYTES
    pts = torch.zeros((n, 3), dtype=torch.float32, device="cuda")
    out = torch.zeros(n, dtype=torch.int32, device="cuda")
    rc = fn(ctypes.c_void_p(pts.data_ptr()), n, 3, 0, ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == kdt.EINVAL
    assert fn(None, 10, 3, 0, ctypes.c_void_p(out.data_ptr()), None) == kdt.EINVAL
