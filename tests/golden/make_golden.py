"""Writes tiny_s6_fp32_oracle.txt: the oracle's outputs on the tiny fp32 S6 workload
(batch 1, d_inner 16, L 256, N 4, seed 0).  Calls only the oracle and the input
generator; the file is a regression snapshot of the oracle, nothing else writes it.

    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_s6_fp32_oracle.txt")


def main():
    w = synth.TINY
    x = synth.make_scan_inputs(w)
    y, h = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"])
    with open(OUT, "w") as f:
        f.write("# oracle outputs, tiny fp32 S6 workload (1 x 16 x 256, N=4, seed 0)\n")
        f.write("# written by tests/golden/make_golden.py (oracle + input generator only)\n")
        f.write("# kind b d index value\n")
        for d in range(w.dim):
            for t in (0, 1, 2, 63, 127, 200, 255):
                f.write("y 0 %d %d %.17g\n" % (d, t, y[0, d, t]))
            for n in range(w.dstate):
                f.write("h 0 %d %d %.17g\n" % (d, n, h[0, d, n]))


if __name__ == "__main__":
    main()
