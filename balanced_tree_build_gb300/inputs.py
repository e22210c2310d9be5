"""Seeded synthetic point clouds (shared by the tests, the bench and smoke()).

This module only draws random numbers: it holds none of the tree method's
arithmetic.  Every workload is float32, AoS (N rows of k coordinates), and is
generated on the host with numpy's PCG64 so that the CUDA build and the CPU
oracle see the same bytes.

Named workloads (sizes, dimensions and split rules of the build's five test
configurations; the seeds are this project's choice except the first):

=================  ===========  ==  ====  =======================================
name               N            k   mode  distribution
=================  ===========  ==  ====  =======================================
uniform_1k         1,000        3   0     U[0,1), seed 0
uniform_pm1_1m     1,048,576    3   0     U[-1,1) as 2u-1, seed 1
mixture_dup_10m    10,000,000   3   0     64-centre Gaussian mixture (sigma
                                          0.01) + 5% exact duplicates, seed 2
quant1024_k8_4m    4,194,304    8   1     floor(u*1024)/1024, seed 3
uniform_100m       100,000,000  3   0     U[0,1), seed 4
=================  ===========  ==  ====  =======================================

mode 0 = split dimension level mod k; mode 1 = widest extent of the domain.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    n: int
    k: int
    mode: int
    dist: str
    seed: int

    def points(self, n: int | None = None) -> np.ndarray:
        """The workload's points; ``n`` draws a smaller sample of the same
        distribution (same seed, so a prefix-free but reproducible sample)."""
        return make_points(self.dist, self.n if n is None else n, self.k, self.seed)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("uniform_1k", 1000, 3, 0, "uniform01", 0),
        Workload("uniform_pm1_1m", 1 << 20, 3, 0, "uniform_pm1", 1),
        Workload("mixture_dup_10m", 10_000_000, 3, 0, "mixture64_dup5", 2),
        Workload("quant1024_k8_4m", 1 << 22, 8, 1, "quant1024", 3),
        Workload("uniform_100m", 100_000_000, 3, 0, "uniform01", 4),
    ]
}


def make_points(dist: str, n: int, k: int, seed: int) -> np.ndarray:
    """Draws an (n, k) float32 C-contiguous array.

    Distributions:
      uniform01       i.i.d. U[0,1) (numpy float32 draws: multiples of 2^-24)
      uniform_pm1     2u - 1 with u as above
      mixture64_dup5  95% of the points from 64 centres ~ U[0,1)^k with
                      N(0, 0.01^2) noise per axis (no clipping), 5% exact
                      copies of uniformly chosen earlier points, then a
                      seeded shuffle of all rows
      quant1024       floor(u * 1024) / 1024, u ~ U[0,1) (exact in float32)
      gaussian        N(0,1)
      all_equal       every coordinate 0.5
      dup_heavy       coordinates drawn from 4 values {0, 0.25, 0.5, 0.75}
      signed_zero     coordinates drawn from {-0.0, +0.0, -1, 1}
      sorted          uniform01, rows sorted by the first coordinate
      reversed        uniform01, rows sorted descending by the first coordinate
      int_grid        small integers 0..15 as floats
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    if n < 0:
        raise ValueError("n must be >= 0")
    if dist == "uniform01":
        return rng.random((n, k), dtype=np.float32)
    if dist == "uniform_pm1":
        u = rng.random((n, k), dtype=np.float32)
        return (np.float32(2.0) * u - np.float32(1.0)).astype(np.float32)
    if dist == "mixture64_dup5":
        n_dup = n // 20
        n_base = n - n_dup
        centres = rng.random((64, k))
        labels = rng.integers(0, 64, size=n_base)
        base = (centres[labels] + rng.normal(0.0, 0.01, size=(n_base, k))).astype(np.float32)
        if n_base == 0:
            return np.zeros((n, k), dtype=np.float32)
        src = rng.integers(0, n_base, size=n_dup)
        pts = np.concatenate([base, base[src]], axis=0)
        order = rng.permutation(n)
        return np.ascontiguousarray(pts[order])
    if dist == "quant1024":
        u = rng.random((n, k))
        return (np.floor(u * 1024.0) / 1024.0).astype(np.float32)
    if dist == "gaussian":
        return rng.standard_normal((n, k), dtype=np.float32)
    if dist == "all_equal":
        return np.full((n, k), 0.5, dtype=np.float32)
    if dist == "dup_heavy":
        vals = np.array([0.0, 0.25, 0.5, 0.75], dtype=np.float32)
        return vals[rng.integers(0, 4, size=(n, k))]
    if dist == "signed_zero":
        vals = np.array([-0.0, 0.0, -1.0, 1.0], dtype=np.float32)
        return vals[rng.integers(0, 4, size=(n, k))]
    if dist == "sorted":
        p = rng.random((n, k), dtype=np.float32)
        return np.ascontiguousarray(p[np.argsort(p[:, 0], kind="stable")])
    if dist == "reversed":
        p = rng.random((n, k), dtype=np.float32)
        return np.ascontiguousarray(p[np.argsort(-p[:, 0], kind="stable")])
    if dist == "int_grid":
        return rng.integers(0, 16, size=(n, k)).astype(np.float32)
    raise ValueError(f"unknown distribution {dist!r}")
