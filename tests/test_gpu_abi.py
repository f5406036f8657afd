"""C-ABI contract on a real device: validation errors are synchronous and
launch nothing (the output buffer keeps its sentinel), status and timing
entry points, path selection."""
import pytest

from protein_pair_representation_gate_b300 import _binding as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def setup():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from synth import make_inputs
    from synth.device import inputs_to_device
    inp = make_inputs("evoformer_256", I=64)
    t = inputs_to_device(inp, "cuda")
    ctx = B.TriAttn(B.TriAttnConfig(128, 4, 32, 64, "bf16"))
    ws = torch.empty(ctx.workspace_bytes(64), dtype=torch.uint8, device="cuda")
    return torch, t, ctx, ws


def _sentinel(torch, like):
    return torch.full_like(like, 7.0)


def test_paths_selected():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    assert B.TriAttn(B.TriAttnConfig(128, 4, 32, 64, "bf16")).path == B.PATH_SM103
    assert B.TriAttn(B.TriAttnConfig(128, 4, 32, 64, "bf16", force_simt=True)).path == B.PATH_SIMT
    assert B.TriAttn(B.TriAttnConfig(32, 4, 8, 64, "f32")).path == B.PATH_SIMT
    assert B.TriAttn(B.TriAttnConfig(64, 2, 16, 64, "bf16")).path == B.PATH_SIMT
    with pytest.raises(B.TriAttnError) as e:
        B.TriAttn(B.TriAttnConfig(64, 2, 24, 64, "bf16"))
    assert e.value.status == B.EUNSUPPORTED


def test_validation_launches_nothing(setup):
    torch, t, ctx, ws = setup
    Z = t["Z"]
    out = _sentinel(torch, Z)
    before = out.clone()
    nbytes = ws.numel()
    cases = [
        dict(node=2),
        dict(I=0),
        dict(I=65),
        dict(Z=Z.data_ptr() + 2),
        dict(out=out.data_ptr() + 2),
        dict(workspace=ws.data_ptr() + 16),
        dict(workspace_bytes=nbytes - 1),
        dict(out=Z.data_ptr()),
        dict(out=ws.data_ptr()),
        dict(weights={**t, "w_q": None}),
        dict(weights={**t, "w_o": t["w_o"].data_ptr() + 2}),
        dict(Z=ws.data_ptr()),                 # input inside the workspace
        dict(mask=out.data_ptr()),             # token mask inside the output
    ]
    want = [B.EINVAL] * 6 + [B.ENOMEM] + [B.EINVAL] * 6
    for kw, st in zip(cases, want):
        args = dict(node=0, I=64, Z=Z, mask=t["mask"], weights=t, workspace=ws, out=out, workspace_bytes=nbytes)
        args.update(kw)
        got = ctx.forward_status(args["node"], args["I"], args["Z"], args["mask"], args["weights"], args["workspace"],
                                 args["out"], None, args["workspace_bytes"])
        assert got == st, (kw, got)
    torch.cuda.synchronize()
    assert torch.equal(out, before)
    assert ctx.status_sync() == B.OK


def test_timing_records_each_kernel(setup):
    torch, t, ctx, ws = setup
    out = torch.empty_like(t["Z"])
    ctx.set_timing(True)
    for node in (0, 1):
        ctx.forward(node, 64, t["Z"], t["mask"], t, ws, out)
    times = ctx.kernel_times()
    ctx.set_timing(False)
    names = [n for n, _ in times]
    assert names.count("sm103_attention") == 2 and names.count("sm103_ln_proj") == 2
    assert all(ms > 0 for _, ms in times)
    assert ctx.kernel_times() == []
    assert ctx.status_sync() == B.OK


def test_output_only_16_byte_aligned(setup):
    """The ABI asks only for a 16-byte aligned out.  The attention epilogue writes
    each output row in 32-byte pieces when out is 32-byte aligned and in 16-byte
    pieces otherwise; both give the same bits (bf16 build, and the fp32-output
    build of the TF32 mode)."""
    torch, t, ctx, ws = setup
    n = t["Z"].numel()
    ref = torch.empty_like(t["Z"])
    buf = torch.empty(n + 8, dtype=t["Z"].dtype, device="cuda")
    off = buf[8:].view_as(t["Z"])                        # 16 bytes past a 256-byte boundary
    assert off.data_ptr() % 32 == 16
    for node in (0, 1):
        ctx.forward(node, 64, t["Z"], t["mask"], t, ws, ref)
        ctx.forward(node, 64, t["Z"], t["mask"], t, ws, off)
        torch.cuda.synchronize()
        assert torch.equal(ref, off), node
    assert ctx.status_sync() == B.OK

    from dataclasses import replace
    from synth import make_inputs
    from synth.device import inputs_to_device
    from synth.workloads import WORKLOADS
    t32 = inputs_to_device(make_inputs(replace(WORKLOADS["evoformer_256"], dtype="f32"), I=64), "cuda")
    ctx32 = B.TriAttn(B.TriAttnConfig(128, 4, 32, 64, "tf32"))
    assert ctx32.path == B.PATH_SM103_TF32
    ws32 = torch.empty(ctx32.workspace_bytes(64), dtype=torch.uint8, device="cuda")
    ref32 = torch.empty_like(t32["Z"])
    buf32 = torch.empty(n + 4, dtype=t32["Z"].dtype, device="cuda")
    off32 = buf32[4:].view_as(t32["Z"])
    assert off32.data_ptr() % 32 == 16
    for node in (0, 1):
        ctx32.forward(node, 64, t32["Z"], t32["mask"], t32, ws32, ref32)
        ctx32.forward(node, 64, t32["Z"], t32["mask"], t32, ws32, off32)
        torch.cuda.synchronize()
        assert torch.equal(ref32, off32), node
    assert ctx32.status_sync() == B.OK


def test_bounded_wait_timeout_is_reported_and_context_recovers(setup):
    """Failure path without a GPU fault: one block's producer skips a stage load,
    its bounded waits run out (~2 s), the launch finishes, status_sync reports
    ETIMEOUT, and the next forward on the same context is correct."""
    import numpy as np
    from tests.gpu_cases import assert_close, oracle_out
    torch, t, ctx, ws = setup
    out = torch.empty_like(t["Z"])
    assert ctx.debug_inject(B.FAULT_SKIP_STAGE) == B.OK
    assert ctx.forward_status(0, 64, t["Z"], t["mask"], t, ws, out) == B.OK
    assert ctx.status_sync() == B.ETIMEOUT
    assert ctx.status_sync() == B.OK                     # the word was cleared
    ctx.forward(0, 64, t["Z"], t["mask"], t, ws, out)
    assert ctx.status_sync() == B.OK
    got = out.float().cpu().numpy().astype(np.float64)
    assert_close(got, oracle_out("evoformer_256", "start", I=64), "bf16", "after recovery")


def test_debug_inject_arguments():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    simt = B.TriAttn(B.TriAttnConfig(32, 4, 8, 64, "f32"))
    assert simt.debug_inject(B.FAULT_SKIP_STAGE) == B.EUNSUPPORTED
    assert simt.debug_inject(B.FAULT_NONE) == B.OK
    tc = B.TriAttn(B.TriAttnConfig(128, 4, 32, 64, "bf16"))
    assert tc.debug_inject(7) == B.EINVAL
    assert tc.debug_inject(B.FAULT_NONE) == B.OK


def test_forward_ex_aliasing_rules(setup):
    """out may equal Z only with the residual; a partial overlap is always EINVAL;
    validation errors launch nothing."""
    torch, t, ctx, ws = setup
    Z = t["Z"].clone()
    before = Z.clone()
    nb = ws.numel()
    assert ctx.forward_status(0, 64, Z, t["mask"], t, ws, Z, None, nb) == B.EINVAL
    pm = torch.ones(64, 64, dtype=torch.uint8, device="cuda")
    assert ctx.forward_status(0, 64, Z, t["mask"], t, ws, Z, None, nb, residual=False, pair_mask=pm) == B.EINVAL
    shifted = Z.data_ptr() + 16 * 128
    assert ctx.forward_status(0, 64, Z, t["mask"], t, ws, shifted, None, nb, residual=True) == B.EINVAL
    torch.cuda.synchronize()
    assert torch.equal(Z, before)
    assert ctx.forward_status(0, 64, Z, t["mask"], t, ws, Z, None, nb, residual=True) == B.OK
    assert ctx.status_sync() == B.OK


def test_large_layernorm_scale_is_finite_or_reported(setup):
    """Intermediates of the sm103 path are f16 (|x| < 65504).  LayerNorm weights
    far beyond a trained model's scale must give either finite output with an OK
    status or the ERANGE status, never silent NaN: gamma = 50 stays inside the
    f16 range (scores then form a hard argmax, so no oracle tolerance applies);
    gamma = 1e5 pushes q, k, v and the pair bias past it."""
    torch, t, ctx, ws = setup
    for scale, want in ((50.0, B.OK), (1e5, B.ERANGE)):
        w = dict(t)
        w["ln_gamma"] = t["ln_gamma"] * scale
        for node in ("start", "end"):
            out = torch.full_like(t["Z"], float("nan"))
            ctx.forward(node, 64, t["Z"], None, w, ws, out)
            st = ctx.status_sync()
            assert st == want, (scale, node, B.status_string(st))
            if st == B.OK:
                assert bool(torch.isfinite(out.float()).all()), (scale, node)
    # the context is usable again at the normal scale
    out = torch.empty_like(t["Z"])
    ctx.forward("start", 64, t["Z"], None, t, ws, out)
    assert ctx.status_sync() == B.OK
    assert bool(torch.isfinite(out.float()).all())
