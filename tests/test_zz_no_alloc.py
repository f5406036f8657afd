"""The allocation-free entry point (tri_attn_forward_static).

tri_attn_forward_static serves callers that cannot allocate device memory
(host callbacks, allocator hooks, plugins whose host owns every allocation):
it takes only inputs and outputs and runs on a library-owned device array.
Its outputs must match the fp64 oracle at the bf16 tolerances and the
context-based entry point's outputs, on two calls in a row (the array keeps
the previous call's contents).  Its validation, status reader and timeout
path are checked too.  This file is named to be collected last.
"""
import numpy as np
import pytest

from tests.gpu_cases import BF16_MAX_ABS, BF16_REL_L2, errors

pytestmark = pytest.mark.gpu


def _need_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def _case(name, I, n_pad):
    from dataclasses import replace
    from synth import make_inputs
    from synth.workloads import WORKLOADS
    return make_inputs(replace(WORKLOADS[name], I=I, n_pad=n_pad))


def test_static_entry_point_matches_oracle_and_forward():
    torch = _need_cuda()
    from oracle import triangle_attention
    from protein_pair_representation_gate_b300 import _binding as B
    from synth.device import inputs_to_device

    calls = [("start", 128, "evoformer_256", 0), ("end", 96, "masked_768", 20)]
    for node, I, name, n_pad in calls:
        inp = _case(name, I, n_pad)
        t = inputs_to_device(inp, "cuda")
        a = inp.oracle_args()
        want = triangle_attention(node, a["Z"], a["mask"], a)
        ctx = B.TriAttn(B.TriAttnConfig(128, 4, 32, I, "bf16"))
        ws = torch.empty(ctx.workspace_bytes(I), dtype=torch.uint8, device="cuda")
        ref = torch.empty_like(t["Z"])
        ctx.forward(node, I, t["Z"], t["mask"], t, ws, ref)
        assert ctx.status_sync() == B.OK
        got = torch.full_like(t["Z"], float("nan"))
        st = B.forward_static(node, I, t["Z"], t["mask"], t, got)
        assert st == B.OK, B.status_string(st)
        assert B.static_status() == B.OK
        g = got.float().cpu().numpy().astype(np.float64)
        r = ref.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(g))
        max_abs, rel = errors(g, want)
        assert max_abs <= BF16_MAX_ABS and rel <= BF16_REL_L2, ("vs oracle", node, I, max_abs, rel)
        max_abs, rel = errors(g, r)
        assert max_abs <= BF16_MAX_ABS and rel <= BF16_REL_L2, ("vs forward", node, I, max_abs, rel)


def test_static_entry_point_rejects_bad_arguments():
    torch = _need_cuda()
    from protein_pair_representation_gate_b300 import _binding as B
    z = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    w = {n: z for n in ("ln_gamma", "ln_beta", "w_q", "w_k", "w_v", "w_g", "w_b", "b_g", "w_o")}
    out = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    assert B.forward_static("start", 129, z, None, w, out) == B.EUNSUPPORTED
    assert B.forward_static("start", 0, z, None, w, out) == B.EINVAL

    # overlaps: out with Z, the token mask inside out; nothing may be launched
    I = 8
    big = torch.zeros(2 * I * I * 128 + 64, dtype=torch.bfloat16, device="cuda")
    Z = big[: I * I * 128]
    out_overlapping = big[I * I * 64: I * I * 64 + I * I * 128]
    sentinel = torch.full((I * I * 128,), 7.0, dtype=torch.bfloat16, device="cuda")
    assert B.forward_static("start", I, Z, None, w, out_overlapping) == B.EINVAL
    mask_in_out = sentinel.view(torch.uint8)[:I]
    assert B.forward_static("start", I, Z, mask_in_out, w, sentinel) == B.EINVAL
    torch.cuda.synchronize()
    assert bool((sentinel == 7.0).all())


def test_static_timeout_is_reported_and_next_call_is_correct():
    torch = _need_cuda()
    from protein_pair_representation_gate_b300 import _binding as B
    from synth.device import inputs_to_device

    I = 64
    inp = _case("evoformer_256", I, 0)
    t = inputs_to_device(inp, "cuda")
    first = torch.empty_like(t["Z"])
    assert B.forward_static("start", I, t["Z"], None, t, first) == B.OK
    assert B.static_status() == B.OK
    assert B.static_debug_inject(7) == B.EINVAL
    assert B.static_debug_inject(B.FAULT_SKIP_STAGE) == B.OK
    broken = torch.empty_like(t["Z"])
    assert B.forward_static("start", I, t["Z"], None, t, broken) == B.OK
    assert B.static_status() == B.ETIMEOUT
    assert B.static_status() == B.OK                  # read once, then cleared
    again = torch.empty_like(t["Z"])
    assert B.forward_static("start", I, t["Z"], None, t, again) == B.OK
    assert B.static_status() == B.OK
    assert torch.equal(again, first)                  # the kernels use no atomics: bitwise repeatable
