"""Write tests/golden/tiny_f32_samples.txt from the oracle (run from the repo root).

The pages print no worked example of the attention, so the stored values are
the oracle's own output on the seeded tiny fp32 workload: a regression pin
that flags any later change of the oracle's arithmetic.  This script calls
only oracle/ and synth/.
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import triangle_attention  # noqa: E402
from synth import make_inputs  # noqa: E402

PAIRS = [(0, 0), (0, 63), (17, 5), (31, 32), (63, 0), (63, 63), (40, 22)]
CHANNELS = [0, 7, 19, 31]


def main():
    inp = make_inputs("tiny_f32")
    a = inp.oracle_args()
    lines = ["# oracle output, tiny fp32 workload (I=64, c_z=32, H=4, d=8, seed 0, no mask)",
             "# written by tests/golden/make_golden.py; columns: node i j channel value"]
    for node in ("start", "end"):
        out = triangle_attention(node, a["Z"], a["mask"], a)
        for i, j in PAIRS:
            for ch in CHANNELS:
                lines.append(f"{node} {i} {j} {ch} {float(out[i, j, ch])!r}")
    with open(os.path.join(HERE, "tiny_f32_samples.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
