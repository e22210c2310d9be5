"""Helpers shared by the GPU tests: run the CUDA build through the C ABI."""
import numpy as np
import torch

import balanced_tree_build_gb300 as kdt
from balanced_tree_build_gb300 import _build

_ready = False


def ensure_library():
    global _ready
    if not _ready:
        _build.build()
        kdt.lib()
        _ready = True


def gpu_build(pts: np.ndarray, mode: int, workspace: bool = True) -> np.ndarray:
    ensure_library()
    d = torch.from_numpy(np.ascontiguousarray(pts, dtype=np.float32)).cuda()
    ws = kdt.alloc_workspace(d.shape[0], d.shape[1], mode) if workspace else None
    perm = kdt.build_tree(d, mode, workspace=ws)
    kdt.check_status()
    return perm.cpu().numpy()
