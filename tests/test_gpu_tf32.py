"""The TF32 mode (fp32 Z, weights and out; tf32 projection operands, f16
attention operands, fp32 accumulation) against the fp64 oracle through the C
ABI on a GPU, at the TF32 tolerance of tests/gpu_cases.py: ragged I on both
nodes, token masks and padding, key chunks, a pair mask with the in-place
residual, non-trivial LayerNorm / gate / output biases, and the CUDA-core
fallback for a shape the TF32 kernels do not cover."""
import numpy as np
import pytest

from tests.gpu_cases import assert_close, errors, oracle_out, run_library
from tests.test_gpu_pair_mask import _pair_mask, _run as run_pair, _want as want_pair

pytestmark = pytest.mark.gpu
NODES = ("start", "end")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("I", [1, 17, 129, 256])
def test_tf32_evoformer_shape(I):
    import protein_pair_representation_gate_b300 as pkg
    res = run_library("evoformer_256", I=I, dtype="tf32")
    assert res["path"] == pkg.PATH_SM103_TF32
    for node in NODES:
        want = oracle_out("evoformer_256", node, I=I, f32=True)
        assert res[node].dtype == np.float64
        max_abs, rel = assert_close(res[node], want, "tf32", f"tf32 I={I} {node}")
        print(f"tf32 I={I} {node}: max abs {max_abs:.3e}, rel L2 {rel:.3e}")


def test_tf32_masked_and_chunked():
    for chunks in (1, 3):
        res = run_library("masked_768", I=200, n_pad=77, key_chunks=chunks, dtype="tf32")
        for node in NODES:
            want = oracle_out("masked_768", node, I=200, n_pad=77, key_chunks=chunks, f32=True)
            assert_close(res[node], want, "tf32", f"tf32 masked chunks={chunks} {node}")
            assert np.all(res[node][:, 200 - 77:] == 0.0) if node == "start" else np.all(res[node][200 - 77:] == 0.0)


def test_tf32_pair_mask_in_place_residual():
    I, n_pad = 160, 10
    pm = _pair_mask(I, seed=6)
    res, dtype = run_pair("masked_768", I, n_pad, pm, in_place=True, dtype="tf32")
    assert dtype == "tf32"
    for node in NODES:
        assert_close(res[node], want_pair("masked_768", node, I, n_pad, pm, residual=True, f32=True), dtype,
                     f"tf32 Z += out {node}")


def test_tf32_affine_params():
    res = run_library("evoformer_256", I=129, affine=True, dtype="tf32")
    for node in NODES:
        assert_close(res[node], oracle_out("evoformer_256", node, I=129, affine=True, f32=True), "tf32",
                     f"tf32 affine {node}")


def test_tf32_more_accurate_than_bf16():
    """The TF32 mode's error against the oracle is below the bf16 path's on the
    same workload (fp32 storage removes the bf16 input and output rounding)."""
    r32 = run_library("evoformer_256", I=256, dtype="tf32", nodes=("start",))
    r16 = run_library("evoformer_256", I=256, nodes=("start",))
    e32 = errors(r32["start"], oracle_out("evoformer_256", "start", I=256, f32=True))
    e16 = errors(r16["start"], oracle_out("evoformer_256", "start", I=256))
    assert e32[1] < e16[1], (e32, e16)


def test_tf32_other_shape_runs_fp32_cuda_cores():
    import protein_pair_representation_gate_b300 as pkg
    res = run_library("tiny_f32", dtype="tf32")
    assert res["path"] == pkg.PATH_SIMT
    for node in NODES:
        assert_close(res[node], oracle_out("tiny_f32", node, f32=True), "f32", f"tf32 fallback {node}")


def test_tf32_path_selection_and_timeout_recovery():
    """Path selection for the TF32 dtype, and the bounded-wait failure path on it:
    one block's producer skips a stage load, the launch ends with ETIMEOUT, and
    the next forward on the same context is correct."""
    import torch
    from protein_pair_representation_gate_b300 import _binding as B
    from synth.device import inputs_to_device
    from tests.gpu_cases import inputs
    assert B.TriAttn(B.TriAttnConfig(128, 4, 32, 64, "tf32")).path == B.PATH_SM103_TF32
    assert B.TriAttn(B.TriAttnConfig(128, 4, 32, 64, "tf32", force_simt=True)).path == B.PATH_SIMT
    assert B.TriAttn(B.TriAttnConfig(64, 2, 16, 64, "tf32")).path == B.PATH_SIMT
    t = inputs_to_device(inputs("evoformer_256", 64, None, False, True), "cuda")
    ctx = B.TriAttn(B.TriAttnConfig(128, 4, 32, 64, "tf32"))
    ws = torch.empty(ctx.workspace_bytes(64), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(t["Z"])
    assert ctx.debug_inject(B.FAULT_SKIP_STAGE) == B.OK
    assert ctx.forward_status(0, 64, t["Z"], t["mask"], t, ws, out) == B.OK
    assert ctx.status_sync() == B.ETIMEOUT
    ctx.forward(0, 64, t["Z"], t["mask"], t, ws, out)
    assert ctx.status_sync() == B.OK
    got = out.cpu().numpy().astype(np.float64)
    assert_close(got, oracle_out("evoformer_256", "start", I=64, f32=True), "tf32", "tf32 after recovery")


def test_tf32_large_layernorm_scale_is_reported():
    """The TF32 mode keeps f16 attention operands: a LayerNorm scale far beyond a
    trained model's pushes them out of range, which the status word reports
    (never silent NaN); the context works again at the normal scale."""
    import torch
    from protein_pair_representation_gate_b300 import _binding as B
    from synth.device import inputs_to_device
    from tests.gpu_cases import inputs
    t = inputs_to_device(inputs("evoformer_256", 64, None, False, True), "cuda")
    ctx = B.TriAttn(B.TriAttnConfig(128, 4, 32, 64, "tf32"))
    ws = torch.empty(ctx.workspace_bytes(64), dtype=torch.uint8, device="cuda")
    w = dict(t)
    w["ln_gamma"] = t["ln_gamma"] * 1e5
    out = torch.full_like(t["Z"], float("nan"))
    ctx.forward("start", 64, t["Z"], None, w, ws, out)
    assert ctx.status_sync() == B.ERANGE
    ctx.forward("start", 64, t["Z"], None, t, ws, out)
    assert ctx.status_sync() == B.OK
    assert bool(torch.isfinite(out).all())


@pytest.mark.slow
def test_tf32_complex_2048_sampled():
    """The TF32 mode on the full I = 2048 workload (the same seeded values in fp32),
    compared on sampled lines: chain boundaries, first and last, both nodes."""
    from tests.gpu_cases import select
    lines = [0, 255, 256, 1023, 2047]
    res = run_library("complex_2048", dtype="tf32")
    for node in NODES:
        got = select(res[node], node, lines)
        want = oracle_out("complex_2048", node, lines=lines, f32=True)
        assert_close(got, want, "tf32", f"tf32 complex_2048 {node} lines={lines}")


def test_tf32_masked_768_sampled():
    """Padded tokens and the amplified pair bias at full size in the TF32 mode."""
    from tests.gpu_cases import select
    lines = [0, 345, 690, 691, 767]
    res = run_library("masked_768", dtype="tf32")
    for node in NODES:
        got = select(res[node], node, lines)
        assert_close(got, oracle_out("masked_768", node, lines=lines, f32=True), "tf32",
                     f"tf32 masked_768 {node} lines={lines}")
        assert np.all(res[node][691:] == 0.0) and np.all(res[node][:, 691:] == 0.0)
