"""Regression pin: the oracle reproduces its stored output on the tiny fp32 workload."""
import os

import numpy as np

from oracle import triangle_attention
from synth import make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiny_f32_samples.txt")


def test_tiny_f32_golden_samples():
    rows = [ln.split() for ln in open(GOLDEN) if ln.strip() and not ln.startswith("#")]
    inp = make_inputs("tiny_f32")
    a = inp.oracle_args()
    outs = {node: triangle_attention(node, a["Z"], a["mask"], a) for node in ("start", "end")}
    assert len(rows) == 56
    for node, i, j, ch, val in rows:
        np.testing.assert_allclose(outs[node][int(i), int(j), int(ch)], float(val), rtol=0, atol=1e-12)
