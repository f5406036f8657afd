"""Run the library on one seeded workload, for timing and profiling (no oracle).

    python -m protein_pair_representation_gate_b300.run_case --workload complex_2048 --I 1024 \
        --nodes start,end --iters 2 [--key-chunks N] [--simt] [--pair-mask DENSITY] [--residual] [--tf32]
    python -m protein_pair_representation_gate_b300.run_case --workload msa_evoformer_512 [--S 512] [--I 256]

Triangle workloads go through tri_attn_forward(_ex); MSA workloads through
tri_attn_msa_forward.  --tf32 runs a triangle workload's seeded values stored in
fp32 in the TF32 mode.  --pair-mask passes a seeded random [I, I] pair mask that
admits each pair with probability DENSITY.  Prints per-kernel CUDA-event times
of the last iteration and the attention kernels' rate in counted TFLOP/s.
"""
from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

PAIR_MASK_STREAM = 13


def _report(op, flops_per_pass: float, passes: int):
    times = op.ctx.kernel_times()
    for name, ms in times:
        print(f"{name:20s} {ms:9.3f} ms")
    att = sum(ms for name, ms in times if "attention" in name)
    if att > 0:
        print(f"attention kernels {att:.3f} ms, {flops_per_pass * passes / (att * 1e-3) / 1e12:.1f} TFLOP/s counted")


def run_triangle(args):
    import numpy as np
    import torch
    import protein_pair_representation_gate_b300 as pkg
    from synth import make_inputs
    from synth.device import inputs_to_device
    from synth.rng import uniform01

    from dataclasses import replace
    from synth.workloads import WORKLOADS
    wl0 = WORKLOADS[args.workload]
    if args.tf32:
        wl0 = replace(wl0, dtype="f32")
    inp = make_inputs(wl0, I=args.I)
    wl = inp.workload
    t = inputs_to_device(inp, "cuda")
    op = pkg.TriangleAttention(wl.c_z, wl.heads, wl.head_dim, wl.I, "tf32" if args.tf32 else wl.dtype,
                               key_chunks=args.key_chunks, force_simt=args.simt)
    pm = None
    if args.pair_mask is not None:
        u = uniform01(wl.seed, PAIR_MASK_STREAM, 0, wl.I * wl.I).reshape(wl.I, wl.I)
        pm = torch.from_numpy((u < args.pair_mask).astype(np.uint8)).cuda()
    out = torch.empty_like(t["Z"])
    nodes = args.nodes.split(",")
    for i in range(args.iters):
        last = i == args.iters - 1
        op.ctx.set_timing(last)
        for node in nodes:
            op(node, t["Z"], t, mask=t["mask"], out=out, pair_mask=pm, residual=args.residual)
        st = op.ctx.status_sync()
        if st != 0:
            raise SystemExit(f"forward failed: {pkg.status_string(st)}")
        if last:
            _report(op, wl.attention_flops(), len(nodes))
    print(f"{args.workload} I={wl.I} nodes={args.nodes} path={['simt', 'sm103', 'sm103_tf32'][op.path]} "
          f"pair_mask={args.pair_mask} residual={args.residual} ok")


def run_msa(args):
    import torch
    import protein_pair_representation_gate_b300 as pkg
    from synth import make_msa_inputs
    from synth.device import msa_inputs_to_device

    inp = make_msa_inputs(args.workload, S=args.S, I=args.I)
    wl = inp.workload
    t = msa_inputs_to_device(inp, "cuda")
    op = pkg.MSARowAttention(wl.c_z, wl.heads, wl.head_dim, wl.I, wl.dtype, key_chunks=args.key_chunks)
    out = torch.empty_like(t["Ms"])
    for i in range(args.iters):
        last = i == args.iters - 1
        op.ctx.set_timing(last)
        op(t["Ms"], t["Z"], t, msa_mask=t["msa_mask"], out=out, residual=args.residual)
        st = op.ctx.status_sync()
        if st != 0:
            raise SystemExit(f"forward failed: {pkg.status_string(st)}")
        if last:
            _report(op, wl.attention_flops(), 1)
    print(f"{args.workload} S={wl.S} I={wl.I} c_m={wl.c_m} residual={args.residual} ok")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="complex_2048")
    ap.add_argument("--I", type=int, default=None)
    ap.add_argument("--S", type=int, default=None, help="MSA rows (MSA workloads)")
    ap.add_argument("--nodes", default="start,end")
    ap.add_argument("--iters", type=int, default=2)
    ap.add_argument("--key-chunks", type=int, default=1)
    ap.add_argument("--simt", action="store_true")
    ap.add_argument("--pair-mask", type=float, default=None, metavar="DENSITY")
    ap.add_argument("--residual", action="store_true")
    ap.add_argument("--tf32", action="store_true", help="fp32 storage, the TF32 mode (triangle workloads)")
    args = ap.parse_args()

    from synth import MSA_WORKLOADS
    if args.workload in MSA_WORKLOADS:
        run_msa(args)
    else:
        run_triangle(args)


if __name__ == "__main__":
    main()
