"""The allocation-free entry point (tri_attn_forward_static) against tri_attn_forward.

tri_attn_forward_static serves callers that cannot allocate device memory
(host callbacks, allocator hooks, plugins whose host owns every allocation):
it takes only inputs and outputs and runs on a library-owned device array.
Its outputs must match the context-based entry point's within the bf16
tolerance of the parity tests, on two calls in a row (the array keeps the
previous call's contents).  This file is named to be collected last.
"""
import numpy as np
import pytest

from tests.gpu_cases import BF16_MAX_ABS, BF16_REL_L2, errors

pytestmark = pytest.mark.gpu


def test_static_entry_point_matches_forward():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from protein_pair_representation_gate_b300 import _binding as B
    from synth import make_inputs
    from synth.device import inputs_to_device

    calls = [("start", 128, "evoformer_256", 0), ("end", 96, "masked_768", 20)]
    for node, I, name, n_pad in calls:
        from dataclasses import replace
        from synth.workloads import WORKLOADS
        inp = make_inputs(replace(WORKLOADS[name], I=I, n_pad=n_pad))
        t = inputs_to_device(inp, "cuda")
        ctx = B.TriAttn(B.TriAttnConfig(128, 4, 32, I, "bf16"))
        ws = torch.empty(ctx.workspace_bytes(I), dtype=torch.uint8, device="cuda")
        ref = torch.empty_like(t["Z"])
        ctx.forward(node, I, t["Z"], t["mask"], t, ws, ref)
        assert ctx.status_sync() == B.OK
        got = torch.full_like(t["Z"], float("nan"))
        st = B.forward_static(node, I, t["Z"], t["mask"], t, got)
        assert st == B.OK, B.status_string(st)
        torch.cuda.synchronize()
        a = got.float().cpu().numpy().astype(np.float64)
        b = ref.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(a))
        max_abs, rel = errors(a, b)
        assert max_abs <= BF16_MAX_ABS and rel <= BF16_REL_L2, (node, I, max_abs, rel)


def test_static_entry_point_rejects_large_I():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from protein_pair_representation_gate_b300 import _binding as B
    z = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    w = {n: z for n in ("ln_gamma", "ln_beta", "w_q", "w_k", "w_v", "w_g", "w_b", "b_g", "w_o")}
    out = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    assert B.forward_static("start", 129, z, None, w, out) == B.EUNSUPPORTED
    assert B.forward_static("start", 0, z, None, w, out) == B.EINVAL
