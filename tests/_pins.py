"""Pins for the CPU oracle: checks against facts fixed by the pages and by
mathematics, each independent of the oracle's own code.

Each pin takes an ``oracle.Oracle`` and raises AssertionError on failure, so
the same battery runs against the real oracle (it must pass) and against the
planted mutants (each must fail at least one pin).

Sources: "GPU-friendly, Parallel, and (Almost-)In-Place Construction of
Left-Balanced k-d Trees" (problem, notation, round-robin, widest-dimension and
worked-example passages); "An Implementation of a Balanced Kd Tree Builder
Using GPUs" (super-key comparison; overview list and build section for the
balanced tree of Brown's builder).
"""
from __future__ import annotations

import os

import numpy as np

from balanced_tree_build_gb300.inputs import make_points

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_worked_example():
    vals = {}
    with open(os.path.join(GOLDEN, "worked_example_10pt.txt")) as f:
        for line in f:
            if line.startswith("#") or ":" not in line:
                continue
            key, rest = line.split(":", 1)
            vals[key.strip()] = rest.strip()
    pts = np.array([[float(v) for v in p.split()] for p in vals["points"].split(";")],
                   dtype=np.float32)
    perm = np.array([int(v) for v in vals["perm"].split()], dtype=np.int32)
    sizes = [int(v) for v in vals["subtree_sizes"].split()]
    return pts, perm, sizes


# ---------------------------------------------------------------------------
# independent helpers (textbook definitions, no oracle code)

def supertuple(pts: np.ndarray, p: int, i: int):
    """(x[p], x[p+1 mod k], ..., x[p-1 mod k], i): the cyclic super key plus
    the input index, compared with Python's tuple order."""
    k = pts.shape[1]
    return tuple(float(pts[i, (p + j) % k]) for j in range(k)) + (i,)


def subtree_count_by_parent_walk(n: int):
    """|S(t)| for every t by tallying each node into all of its ancestors
    (parent(i) = (i-1)//2)."""
    cnt = [0] * n
    for i in range(n):
        a = i
        while True:
            cnt[a] += 1
            if a == 0:
                break
            a = (a - 1) // 2
    return cnt


def subtree_closed_form(n: int, s: int) -> int:
    """Closed form of the left-balanced subtree size (derived from the shape:
    levels 0..L-2 full, the last level filled from the left)."""
    if s >= n:
        return 0
    L = n.bit_length()  # numLevels(n)
    l = (s + 1).bit_length() - 1  # level(s)
    M = n - ((1 << (L - 1)) - 1)
    A = (1 << (L - 1 - l)) - 1
    B = 1 << (L - 1 - l)
    j = s - ((1 << l) - 1)
    return A + min(max(M - j * B, 0), B)


def inorder(n: int):
    out = []
    stack = []
    i = 0
    while stack or i < n:
        while i < n:
            stack.append(i)
            i = 2 * i + 1
        i = stack.pop()
        out.append(i)
        i = 2 * i + 2
    return out


# ---------------------------------------------------------------------------
# pins

def pin_worked_example(o):
    pts, perm, sizes = load_worked_example()
    got = o.build_tree(pts, mode=0)
    assert np.array_equal(got, perm), (got, perm)
    assert [o.subtree_count(10, s) for s in range(10)] == sizes
    cnt, first = o.brute_force(pts, mode=0)
    assert cnt == 1 and np.array_equal(first, perm)


def pin_less_is_tuple_order(o):
    for k in (1, 2, 3, 4):
        for dist in ("dup_heavy", "int_grid", "signed_zero"):
            pts = make_points(dist, 24, k, seed=11 + k)
            for p in range(k):
                for a in range(24):
                    for b in range(24):
                        want = supertuple(pts, p, a) < supertuple(pts, p, b)
                        assert o.less(pts, p, a, b) == want, (k, dist, p, a, b)


def pin_widest_dim_is_first_argmax(o):
    rng = np.random.default_rng(5)
    for k in (1, 2, 3, 5, 8):
        for _ in range(300):
            lo = (np.floor(rng.random(k) * 4) / 4).astype(np.float32)
            hi = lo + (np.floor(rng.random(k) * 4) / 4).astype(np.float32)
            ext = (hi - lo).astype(np.float32)
            assert o.widest_dim(lo, hi) == int(np.argmax(ext)), (lo, hi)


def pin_subtree_count(o):
    for n in list(range(1, 130)) + [255, 256, 257, 300]:
        want = subtree_count_by_parent_walk(n)
        got = [o.subtree_count(n, t) for t in range(n)]
        assert got == want, n
        assert o.subtree_count(n, n) == 0
    assert o.num_levels(1) == 1 and o.num_levels(2) == 2 and o.num_levels(1000) == 10


def pin_subtree_closed_form_large(o):
    rng = np.random.default_rng(9)
    for n in [2**20, 2**20 - 1, 2**20 + 1, 10_000_000, 100_000_000, 2**31 - 1]:
        L = n.bit_length()
        assert o.num_levels(n) == L
        for _ in range(200):
            s = int(rng.integers(0, n))
            assert o.subtree_count(n, s) == subtree_closed_form(n, s), (n, s)


def pin_brute_force_unique(o, sizes=range(1, 9), ks=(1, 2, 3), modes=(0, 1)):
    seed = 100
    for n in sizes:
        for k in ks:
            for mode in modes:
                for dist in ("uniform01", "dup_heavy", "all_equal", "int_grid", "signed_zero"):
                    seed += 1
                    pts = make_points(dist, n, k, seed)
                    cnt, first = o.brute_force(pts, mode)
                    assert cnt == 1, (n, k, mode, dist, cnt)
                    got = o.build_tree(pts, mode)
                    assert np.array_equal(got, first), (n, k, mode, dist, got, first)


def pin_k1_inorder_sorted(o):
    for n, dist in [(1, "uniform01"), (2, "dup_heavy"), (17, "int_grid"), (1000, "dup_heavy"),
                    (4097, "uniform01"), (3000, "signed_zero")]:
        pts = make_points(dist, n, 1, seed=n)
        perm = o.build_tree(pts, mode=0)
        order = np.lexsort((np.arange(n), pts[:, 0]))  # by x, then index
        assert np.array_equal(perm[inorder(n)], order), (n, dist)


def pin_perfect_tree_root_is_median(o):
    for m in (3, 7, 11):
        n = (1 << m) - 1
        pts = make_points("uniform01", n, 3, seed=m)
        perm = o.build_tree(pts, mode=0)
        assert pts[perm[0], 0] == np.median(pts[:, 0])


def pin_cyclic_tiebreak_top_nodes(o):
    """Root and node 1 picked by numpy lexsort on explicit key columns."""
    for dist in ("dup_heavy", "int_grid", "quant1024"):
        n, k = 500, 3
        pts = make_points(dist, n, k, seed=77)
        perm = o.build_tree(pts, mode=0)
        idx = np.arange(n)
        order0 = np.lexsort((idx, pts[:, 2], pts[:, 1], pts[:, 0]))
        m = subtree_closed_form(n, 1)
        assert perm[0] == order0[m]
        left = order0[:m]
        order1 = left[np.lexsort((left, pts[left, 0], pts[left, 2], pts[left, 1]))]
        assert perm[1] == order1[subtree_closed_form(n, 3)]
        right = order0[m + 1:]
        order2 = right[np.lexsort((right, pts[right, 0], pts[right, 2], pts[right, 1]))]
        assert perm[2] == order2[subtree_closed_form(n, 5)]


def pin_widest_root_and_children(o):
    """Widest mode: root dimension = first argmax of the bounding-box extent;
    children domains are the root box cut at the root's split coordinate."""
    rng = np.random.default_rng(3)
    for trial in range(6):
        n, k = 400, 4
        pts = make_points("quant1024", n, k, seed=300 + trial)
        scale = np.ones(k, dtype=np.float32)
        scale[trial % k] = 3.0  # make one dimension clearly widest
        if trial >= 4:
            scale[:] = 1.0  # extents tie: the lowest dimension must win
        pts = (pts * scale).astype(np.float32)
        perm = o.build_tree(pts, mode=1)
        lo, hi = pts.min(axis=0), pts.max(axis=0)
        d0 = int(np.argmax((hi - lo).astype(np.float32)))
        idx = np.arange(n)
        keys = [pts[:, (d0 + j) % k] for j in range(k)]
        order0 = np.lexsort([idx] + keys[::-1])
        m = subtree_closed_form(n, 1)
        assert perm[0] == order0[m], trial
        split = pts[perm[0], d0]
        for child, members, side in ((1, order0[:m], "hi"), (2, order0[m + 1:], "lo")):
            clo, chi = lo.copy(), hi.copy()
            (chi if side == "hi" else clo)[d0] = split
            d1 = int(np.argmax((chi - clo).astype(np.float32)))
            ck = [pts[members, (d1 + j) % k] for j in range(k)]
            oc = members[np.lexsort([members] + ck[::-1])]
            assert perm[child] == oc[subtree_closed_form(n, 2 * child + 1)], (trial, child)
    del rng


def pin_verifier_rejects(o):
    rng = np.random.default_rng(8)
    for mode in (0, 1):
        pts = make_points("dup_heavy", 300, 3, seed=21 + mode)
        perm = o.build_tree(pts, mode)
        ok, _ = o.verify(pts, perm, mode)
        assert ok
        for _ in range(40):
            a, b = rng.choice(300, size=2, replace=False)
            bad = perm.copy()
            bad[a], bad[b] = bad[b], bad[a]
            ok, node = o.verify(pts, bad, mode)
            assert not ok
        dup = perm.copy()
        dup[5] = dup[6]
        ok, node = o.verify(pts, dup, mode)
        assert not ok and node == -1


# ---------------------------------------------------------------------------
# the balanced (median-split) tree of Brown's builder: "An Implementation of
# a Balanced Kd Tree Builder Using GPUs", overview list (sort, take the
# median, partition the other arrays, cycle through the coordinates) and
# build section (per-level median store, children of entry j at 2j, 2j+1).

def balanced_shape_by_sizes(n: int) -> set:
    """Occupied heap slots of the balanced tree of n points, from the split
    rule alone: the lower side gets floor((m-1)/2) of a subtree's m points."""
    occ, stack = set(), [(0, n)]
    while stack:
        s, m = stack.pop()
        if m == 0:
            continue
        occ.add(s)
        left = (m - 1) // 2
        stack += [(2 * s + 1, left), (2 * s + 2, m - 1 - left)]
    return occ


def heap_inorder(slots: np.ndarray) -> list:
    """Occupied slots' values in in-order (left subtree, node, right subtree)."""
    out, stack, s = [], [], 0
    while stack or (s < slots.size and slots[s] >= 0):
        while s < slots.size and slots[s] >= 0:
            stack.append(s)
            s = 2 * s + 1
        s = stack.pop()
        out.append(int(slots[s]))
        s = 2 * s + 2
    return out


def lexsort_super(pts: np.ndarray, ids: np.ndarray, p: int) -> np.ndarray:
    """ids ordered by (x[p], x[p+1 mod k], ..., input index) with numpy's
    lexsort on explicit key columns (the last key is the primary one)."""
    k = pts.shape[1]
    keys = [ids] + [pts[ids, (p + j) % k] for j in reversed(range(k))]
    return ids[np.lexsort(keys)]


def pin_balanced_brute_force_unique(o, sizes=range(1, 9), ks=(1, 2, 3)):
    for n in sizes:
        for k in ks:
            for dist in ("uniform01", "dup_heavy", "all_equal", "int_grid"):
                pts = make_points(dist, n, k, seed=100 * n + k)
                cnt, first = o.brute_force_balanced(pts)
                assert cnt == 1, (n, k, dist, cnt)
                assert np.array_equal(o.build_balanced(pts), first), (n, k, dist)


def pin_balanced_shape(o):
    for n in list(range(1, 130)) + [1000, 4095, 4096, 4097, 65537]:
        pts = make_points("uniform01", n, 2, seed=n)
        slots = o.build_balanced(pts)
        assert slots.size == 2 ** n.bit_length() - 1
        assert set(np.nonzero(slots >= 0)[0].tolist()) == balanced_shape_by_sizes(n), n
        assert np.array_equal(np.sort(slots[slots >= 0]), np.arange(n))


def pin_balanced_k1_inorder_sorted(o):
    for n in (1, 2, 3, 10, 31, 32, 100, 1000):
        for dist in ("uniform01", "dup_heavy"):
            pts = make_points(dist, n, 1, seed=n + 7)
            want = lexsort_super(pts, np.arange(n), 0)
            assert heap_inorder(o.build_balanced(pts)) == want.tolist(), (n, dist)


def pin_balanced_root_and_children(o):
    for n, dist, k in [(101, "dup_heavy", 3), (1000, "uniform01", 2), (64, "int_grid", 3), (7, "all_equal", 2)]:
        pts = make_points(dist, n, k, seed=n)
        slots = o.build_balanced(pts)
        order0 = lexsort_super(pts, np.arange(n), 0)
        m = (n - 1) // 2
        assert slots[0] == order0[m], (n, dist)
        for part, slot in ((order0[:m], 1), (order0[m + 1:], 2)):
            if part.size == 0:
                continue
            o1 = lexsort_super(pts, np.sort(part), 1 % k)
            assert slots[slot] == o1[(part.size - 1) // 2], (n, dist, slot)


def pin_balanced_verifier_rejects(o):
    pts = make_points("dup_heavy", 300, 3, seed=3)
    slots = o.build_balanced(pts)
    assert o.verify_balanced(pts, slots)[0]
    occ = np.nonzero(slots >= 0)[0]
    bad = slots.copy()
    bad[[occ[5], occ[200]]] = bad[[occ[200], occ[5]]]
    assert not o.verify_balanced(pts, bad)[0]
    moved = slots.copy()
    hole = int(np.nonzero(slots < 0)[0][0])
    moved[hole], moved[occ[-1]] = moved[occ[-1]], -1
    assert not o.verify_balanced(pts, moved)[0]


ALL_PINS = [
    pin_worked_example,
    pin_less_is_tuple_order,
    pin_widest_dim_is_first_argmax,
    pin_subtree_count,
    pin_subtree_closed_form_large,
    pin_brute_force_unique,
    pin_k1_inorder_sorted,
    pin_perfect_tree_root_is_median,
    pin_cyclic_tiebreak_top_nodes,
    pin_widest_root_and_children,
    pin_verifier_rejects,
    pin_balanced_brute_force_unique,
    pin_balanced_shape,
    pin_balanced_k1_inorder_sorted,
    pin_balanced_root_and_children,
    pin_balanced_verifier_rejects,
]
