"""Run tri_attn_forward on one seeded workload, for profiling (no oracle).

    python -m protein_pair_representation_gate_b300.run_case --workload complex_2048 --I 1024 \
        --nodes start,end --iters 2 [--key-chunks N] [--simt]

Prints per-kernel CUDA-event times of the last iteration.
"""
from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="complex_2048")
    ap.add_argument("--I", type=int, default=None)
    ap.add_argument("--nodes", default="start,end")
    ap.add_argument("--iters", type=int, default=2)
    ap.add_argument("--key-chunks", type=int, default=1)
    ap.add_argument("--simt", action="store_true")
    args = ap.parse_args()

    import torch
    import protein_pair_representation_gate_b300 as pkg
    from synth import make_inputs
    from synth.device import inputs_to_device

    inp = make_inputs(args.workload, I=args.I)
    wl = inp.workload
    t = inputs_to_device(inp, "cuda")
    op = pkg.TriangleAttention(wl.c_z, wl.heads, wl.head_dim, wl.I, wl.dtype, key_chunks=args.key_chunks,
                               force_simt=args.simt)
    out = torch.empty_like(t["Z"])
    for i in range(args.iters):
        last = i == args.iters - 1
        op.ctx.set_timing(last)
        for node in args.nodes.split(","):
            op(node, t["Z"], t, mask=t["mask"], out=out)
        st = op.ctx.status_sync()
        if st != 0:
            raise SystemExit(f"forward failed: {pkg.status_string(st)}")
        if last:
            for name, ms in op.ctx.kernel_times():
                print(f"{name:20s} {ms:9.3f} ms")
    print(f"{args.workload} I={wl.I} nodes={args.nodes} path={['simt', 'sm103'][op.path]} ok")


if __name__ == "__main__":
    main()
