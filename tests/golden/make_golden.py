"""Writes the text fixtures in this folder from the formulas the pages print.

Nothing here calls the CUDA library; the fixtures are the pages' own worked
examples evaluated as printed, so the oracle is checked against them rather
than against itself.

* ldmatrix_x2_interleaved.txt -- "ldmatrix / stmatrix", section "Example:
  interleaved shared rows and register slots 0, 2, 8, 10": shared data
  x = arange(128) viewed as (16, 4, 2) uint32; every lane starts with twelve
  sentinel words 4294966519 (the bit pattern of int32 -777); two .x2
  issues then write slot 8*k + 2*matrix of lane l with
  x[2*(l//4) + matrix, l%4, k].
* add_one_2x32x3x4.txt -- "Tile Operands and Execution", section "A Load,
  Compute, and Store Example": A = arange(768) as float32 (2, 32, 3, 4);
  the result is A + 1.  Stored as the flat list of expected values.

Two fixtures here are written by hand, not by this script, because the
pages state them as rules rather than as arrays:

* block_scale_tmem_slots.txt -- "tcgen05.mma", section "Weight-stationary and
  block scaling": TMEM lane and byte column of a scale row's factor, with its
  four replicas, for selected rows.
* ldmatrix_x2_address_providers.txt -- "ldmatrix / stmatrix", the operand
  example's sentence on which lanes provide which row addresses.

Run: python tests/golden/make_golden.py
"""
import os

HERE = os.path.dirname(os.path.abspath(__file__))
SENTINEL = 4294966519


def ldmatrix_x2_interleaved():
    x = [[[2 * (4 * r + w) + k for k in range(2)] for w in range(4)] for r in range(16)]
    rows = []
    for lane in range(32):
        words = [SENTINEL] * 12
        for k in range(2):
            for matrix in range(2):
                words[8 * k + 2 * matrix] = x[2 * (lane // 4) + matrix][lane % 4][k]
        rows.append(words)
    return rows


def main():
    with open(os.path.join(HERE, "ldmatrix_x2_interleaved.txt"), "w") as f:
        f.write("# ldmatrix / stmatrix -- Example: interleaved shared rows and register\n")
        f.write("# slots 0, 2, 8, 10.  x = arange(128) as uint32 (16, 4, 2); one row per\n")
        f.write("# lane, twelve register words each; sentinel 4294966519 = int32(-777).\n")
        for words in ldmatrix_x2_interleaved():
            f.write(" ".join(str(v) for v in words) + "\n")
    with open(os.path.join(HERE, "add_one_2x32x3x4.txt"), "w") as f:
        f.write("# Tile Operands and Execution -- A Load, Compute, and Store Example.\n")
        f.write("# A = arange(768) as float32 (2, 32, 3, 4); expected B = A + 1, flat.\n")
        vals = [float(v + 1) for v in range(768)]
        for i in range(0, 768, 12):
            f.write(" ".join(repr(v) for v in vals[i:i + 12]) + "\n")


if __name__ == "__main__":
    main()
