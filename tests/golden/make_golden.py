"""Writes the stored expected values under tests/golden/ by calling only the oracle.

Run from the repository root:  python tests/golden/make_golden.py

int_tile_bf16.txt -- the pages' single-tile workload shape (BF16 M=32, N=64,
K=128, two splits of 64) on integer operands in [-8, 8] (seed 3), where every
product and sum is exact; it freezes the oracle's P[2,32,64] and O[32,64].
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import splitk_inputs as gen  # noqa: E402


def main():
    ops = gen.integers(32, 64, 128, "bf16", seed=3)
    P, _ = oracle.partials(ops.A, ops.B, "bf16", 128, 2, 64)
    O, _ = oracle.output(ops.A, ops.B, "bf16")
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "int_tile_bf16.txt")
    with open(out, "w") as f:
        f.write("# BF16 M=32 N=64 K=128 splits=2 kps=64; integer operands in [-8,8], seed 3\n")
        f.write("# written by tests/golden/make_golden.py from the oracle\n")
        for s in range(2):
            f.write(f"P{s}\n")
            for row in P[s].astype(np.int64):
                f.write(" ".join(str(v) for v in row) + "\n")
        f.write("O\n")
        for row in O.astype(np.int64):
            f.write(" ".join(str(v) for v in row) + "\n")


if __name__ == "__main__":
    main()
