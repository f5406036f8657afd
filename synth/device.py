"""Copy one workload's seeded inputs to torch tensors (no arithmetic of the method).

bf16 storage arrays (uint16 bit patterns) become torch.bfloat16 tensors with
the very same bits; float32 arrays stay float32.
"""
from __future__ import annotations

import numpy as np
import torch

from .workloads import Inputs

TENSORS = ("Z", "w_q", "w_k", "w_v", "w_g", "w_b", "w_o", "ln_gamma", "ln_beta", "b_g", "b_o")


def to_torch(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a))


def inputs_to_device(inp: Inputs, device="cuda", pin: bool = False) -> dict:
    """dict of tensors keyed like the library's weights struct, plus "Z" and "mask"."""
    out = {}
    for n in TENSORS + ("mask",):
        t = to_torch(getattr(inp, n))
        if device == "cpu":
            out[n] = t.pin_memory() if pin else t.clone()
        else:
            out[n] = t.to(device)
    return out


def msa_inputs_to_device(inp, device="cuda") -> dict:
    """MSA inputs as tensors keyed like tri_attn_msa_weights, plus "Ms", "Z" and "msa_mask"."""
    return {n: to_torch(getattr(inp, n)).to(device) for n in inp.TENSORS + ("msa_mask",)}
