"""The largest build the ABI accepts: N = 2^31 - 1 points (GPU required,
~100 GB of device memory; skipped when the device has less free).

The points are drawn on the device (the oracle cannot build 2^31 points in
test time), so the check is the GPU verifier: perm is a permutation and every
node satisfies the tree conditions against every ancestor, which by
uniqueness of the tree equals agreement with the oracle.  k = 2 keeps the
memory down while the first coordinate carries heavy ties (float32 uniform
draws take 2^24 values), so the global levels resolve large candidate sets and
the finisher hands crowded tiles to the select finisher."""
import pytest
import torch

import balanced_tree_build_gb300 as kdt
from gpu_util import ensure_library

pytestmark = pytest.mark.gpu

N_MAX = 2**31 - 1


def test_build_at_the_size_limit():
    ensure_library()
    k, mode = 2, 0
    need = kdt.workspace_bytes(N_MAX, k, mode) + N_MAX * (4 * k + 4) + (8 << 30)
    free, _ = torch.cuda.mem_get_info()
    if free < need:
        pytest.skip(f"needs {need / 1e9:.0f} GB free on the device, has {free / 1e9:.0f} GB")
    g = torch.Generator(device="cuda")
    g.manual_seed(31)
    pts = torch.rand((N_MAX, k), generator=g, device="cuda", dtype=torch.float32)
    ws = kdt.alloc_workspace(N_MAX, k, mode)
    perm = kdt.build_tree(pts, mode, workspace=ws)
    kdt.check_status()
    del ws
    torch.cuda.empty_cache()
    assert kdt.verify_tree(pts, perm, mode)
    # the root is the point of rank ss(1) = 2^30 - 1 + min(M, 2^30) under <_0;
    # its first coordinate splits the others accordingly
    root = pts[perm[0].long()]
    below = (pts[:, 0] < root[0]).sum().item()
    assert below <= 2**31 - 1 - 2**30
