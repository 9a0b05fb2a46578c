"""Writes the fixtures in this folder.

  varlen_group_counts_g64_m32768_seed0.txt
      the per-group row counts that the seeded varlen-M workload generator
      draws (64 groups, 32768 rows, 4 empty groups, seed 0).  It is an input
      fixture: it pins the generator's output across machines and library
      versions.
  fastdivmod_params.txt
      (divisor, multiplier, shift) from the oracle's FastDivmod for the
      divisors the workloads' tile grids use, plus edge divisors.

Run from the repository root:  python tests/golden/write_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import fastdivmod  # noqa: E402
from grouped_gemm_epilogues_gb300 import workloads  # noqa: E402


def main():
    sizes = workloads.group_sizes(32768, 64, 4, 0)
    with open(os.path.join(HERE, "varlen_group_counts_g64_m32768_seed0.txt"), "w") as f:
        f.write("# rows per group, seed 0 (written by write_golden.py)\n")
        f.write(" ".join(str(int(s)) for s in sizes) + "\n")
    divisors = sorted({1, 2, 3, 5, 6, 7, 8, 12, 16, 24, 32, 48, 64, 128, 256, 512, 1000,
                       65535, 65536, 65537, 2 ** 30 + 1, 2 ** 31 - 1,
                       1 * 2, 2 * 2, 16 * 16, 64 * 32, 32 * 64, 8 * 32, 8 * 16, 8 * 6})
    with open(os.path.join(HERE, "fastdivmod_params.txt"), "w") as f:
        f.write("# divisor multiplier shift (oracle FastDivmod; written by write_golden.py)\n")
        for d in divisors:
            _, m, s = fastdivmod.create(d)
            f.write(f"{d} {m} {s}\n")


if __name__ == "__main__":
    main()
