"""Writes the stored expected values under tests/golden/ from the CPU oracle.

Calls only ``oracle`` (exhaustive search and the recursive builder); nothing
here comes from the CUDA library.  Run from the repository root:

    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402

# The ten int2 points of the worked example in "GPU-friendly, Parallel, and
# (Almost-)In-Place Construction of Left-Balanced k-d Trees" (example
# section).  The page prints the points; its step-by-step tables did not
# survive, so the expected tree is found here by exhaustive search over all
# 10! orderings under the tree conditions.
POINTS = [(10, 15), (46, 63), (68, 21), (40, 33), (25, 54),
          (15, 43), (44, 58), (45, 40), (62, 69), (53, 67)]


def main():
    o = oracle.get()
    pts = np.array(POINTS, dtype=np.float32)
    count, perm = o.brute_force(pts, mode=0)
    assert count == 1, count
    sizes = [o.subtree_count(len(POINTS), s) for s in range(len(POINTS))]
    path = os.path.join(HERE, "worked_example_10pt.txt")
    with open(path, "w") as f:
        f.write("# Worked example: \"GPU-friendly, Parallel, and (Almost-)In-Place Construction of\n")
        f.write("# Left-Balanced k-d Trees\", example section.  The page prints the ten int2 points;\n")
        f.write("# its step tables are missing from the extracted text.  k = 2, split dimension\n")
        f.write("# level mod 2.  'perm' (level-order node -> input index) was written by\n")
        f.write("# tests/golden/make_golden.py from an exhaustive search over all 10! orderings\n")
        f.write("# (exactly one satisfies the tree conditions); it also matches a hand trace of\n")
        f.write("# the tag method.  'subtree_sizes' are |S(s)| for s = 0..9 of the 10-node tree.\n")
        f.write("points: " + "; ".join(f"{x} {y}" for x, y in POINTS) + "\n")
        f.write("perm: " + " ".join(str(int(v)) for v in perm) + "\n")
        f.write("subtree_sizes: " + " ".join(str(v) for v in sizes) + "\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
