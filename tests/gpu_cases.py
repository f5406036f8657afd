"""Helpers of the GPU parity tests: run the library through the C-ABI on one
workload and compare with the fp64 oracle at the stated tolerances."""
from __future__ import annotations

import functools

import numpy as np

from oracle import pair_bias, triangle_attention
from synth import make_inputs, with_affine_params

# Tolerances: fp32 path max-abs 1e-4; bf16 inputs with fp32 accumulation
# max-abs 2e-2 and relative L2 error 5e-3 over the compared outputs.
F32_MAX_ABS = 1e-4
BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 5e-3
# TF32 mode (fp32 storage; tf32 projection operands, f16 attention operands, fp32
# accumulation and output): the bf16 bound scaled by the ratio of the coarsest
# rounding on each path -- tf32 truncation of the stored fp32 inputs (relative
# error < 2^-10) against bf16 rounding of the stored inputs and the output
# (< 2^-9) -- i.e. halved.
TF32_MAX_ABS = BF16_MAX_ABS / 2
TF32_REL_L2 = BF16_REL_L2 / 2


@functools.lru_cache(maxsize=4)
def inputs(name: str, I: int | None = None, n_pad: int | None = None, affine: bool = False, f32: bool = False):
    """Seeded inputs of a workload; f32=True stores them in fp32 (the TF32 mode's storage)."""
    from dataclasses import replace
    from synth.workloads import WORKLOADS
    wl = WORKLOADS[name]
    if f32:
        wl = replace(wl, dtype="f32")
    if I is not None:
        wl = replace(wl, I=I, n_pad=min(wl.n_pad if n_pad is None else n_pad, I))
    elif n_pad is not None:
        wl = replace(wl, n_pad=n_pad)
    inp = make_inputs(wl)
    return with_affine_params(inp) if affine else inp


@functools.lru_cache(maxsize=2)
def oracle_state(name, I=None, n_pad=None, affine=False, f32=False):
    inp = inputs(name, I, n_pad, affine, f32)
    a = inp.oracle_args()
    return a, pair_bias(a["Z"], a["ln_gamma"], a["ln_beta"], a["w_b"])


def oracle_out(name, node, lines=None, I=None, n_pad=None, key_chunks=1, affine=False, f32=False):
    a, bias = oracle_state(name, I, n_pad, affine, f32)
    return triangle_attention(node, a["Z"], a["mask"], a, lines=lines, key_chunks=key_chunks, bias=bias)


def run_library(name, nodes=("start", "end"), I=None, n_pad=None, key_chunks=1, force_simt=False, repeat=1,
                affine=False, dtype=None):
    """dtype "tf32" runs the fp32-stored inputs in the TF32 mode."""
    """Outputs of tri_attn_forward (through the C-ABI) as float64 numpy arrays, per node."""
    import torch
    import protein_pair_representation_gate_b300 as pkg
    from synth.device import inputs_to_device

    inp = inputs(name, I, n_pad, affine, dtype == "tf32")
    wl = inp.workload
    t = inputs_to_device(inp, "cuda")
    op = pkg.TriangleAttention(wl.c_z, wl.heads, wl.head_dim, wl.I, dtype or wl.dtype, key_chunks=key_chunks,
                               force_simt=force_simt)
    res = {}
    for node in nodes:
        outs = []
        for _ in range(repeat):
            out = op(node, t["Z"], t, mask=t["mask"])
            st = op.ctx.status_sync()
            assert st == 0, pkg.status_string(st)
            outs.append(out.float().cpu().numpy().astype(np.float64) if out.dtype != torch.float32
                        else out.cpu().numpy().astype(np.float64))
        res[node] = outs if repeat > 1 else outs[0]
    res["path"] = op.path
    del t, op
    torch.cuda.empty_cache()
    return res


def select(out, node, lines):
    return out[lines] if node == "start" else out[:, lines]


def errors(got, want):
    diff = got - want
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    den = float(np.sqrt((want ** 2).sum()))
    rel = float(np.sqrt((diff ** 2).sum()) / den) if den > 0 else float(np.sqrt((diff ** 2).sum()))
    return max_abs, rel


def assert_close(got, want, dtype, what=""):
    max_abs, rel = errors(got, want)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if dtype == "f32":
        assert max_abs <= F32_MAX_ABS, f"{what}: max abs {max_abs:.3e} > {F32_MAX_ABS}"
    elif dtype == "tf32":
        assert max_abs <= TF32_MAX_ABS and rel <= TF32_REL_L2, \
            f"{what}: max abs {max_abs:.3e} (<= {TF32_MAX_ABS}), rel L2 {rel:.3e} (<= {TF32_REL_L2})"
    else:
        assert max_abs <= BF16_MAX_ABS and rel <= BF16_REL_L2, \
            f"{what}: max abs {max_abs:.3e} (<= {BF16_MAX_ABS}), rel L2 {rel:.3e} (<= {BF16_REL_L2})"
    return max_abs, rel
