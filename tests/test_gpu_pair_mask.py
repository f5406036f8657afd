"""Pair mask M[I, I] and the residual update (tri_attn_forward_ex) against the
fp64 oracle, on both paths; through the C ABI on a GPU."""
import numpy as np
import pytest

from oracle import triangle_attention
from tests.gpu_cases import assert_close, inputs, oracle_state

pytestmark = pytest.mark.gpu
NODES = ("start", "end")


def _pair_mask(I, seed=3, p_valid=0.8):
    rng = np.random.default_rng(seed)
    return rng.random((I, I)) < p_valid


def _run(name, I, n_pad, pm, nodes=NODES, key_chunks=1, force_simt=False, residual=False, in_place=False,
         dtype=None):
    import torch
    import protein_pair_representation_gate_b300 as pkg
    from synth.device import inputs_to_device
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    inp = inputs(name, I, n_pad, False, dtype == "tf32")
    wl = inp.workload
    t = inputs_to_device(inp, "cuda")
    op = pkg.TriangleAttention(wl.c_z, wl.heads, wl.head_dim, wl.I, dtype or wl.dtype, key_chunks=key_chunks,
                               force_simt=force_simt)
    dpm = torch.from_numpy(pm.astype(np.uint8)).cuda() if pm is not None else None
    res = {}
    for node in nodes:
        if in_place:
            z = t["Z"].clone()
            op(node, z, t, mask=t["mask"], out=z, pair_mask=dpm, residual=True)
            out = z
        else:
            out = op(node, t["Z"], t, mask=t["mask"], pair_mask=dpm, residual=residual)
        assert op.ctx.status_sync() == 0
        res[node] = out.float().cpu().numpy().astype(np.float64)
    return res, dtype or wl.dtype


def _want(name, node, I, n_pad, pm, key_chunks=1, residual=False, f32=False):
    a, bias = oracle_state(name, I, n_pad, False, f32)
    return triangle_attention(node, a["Z"], a["mask"], a, key_chunks=key_chunks, bias=bias, pair_mask=pm,
                              residual=residual)


@pytest.mark.parametrize("I, n_pad", [(200, 17), (64, 0)])
def test_pair_mask_tensor_core_path(I, n_pad):
    pm = _pair_mask(I)
    res, dtype = _run("masked_768", I, n_pad, pm)
    valid = (np.arange(I) < I - n_pad)
    for node in NODES:
        assert_close(res[node], _want("masked_768", node, I, n_pad, pm), dtype, f"pair mask I={I} {node}")
        masked = ~(pm & valid[:, None] & valid[None, :])
        assert np.all(res[node][masked] == 0.0)


def test_pair_mask_with_key_chunks():
    """Key chunks of 72 start off a 64-key boundary, so tiles read two mask words."""
    I, n_pad = 200, 9
    pm = _pair_mask(I, seed=4)
    res, dtype = _run("masked_768", I, n_pad, pm, key_chunks=3)
    for node in NODES:
        assert_close(res[node], _want("masked_768", node, I, n_pad, pm, key_chunks=3), dtype, f"chunked {node}")


def test_pair_mask_line_fully_masked():
    I = 96
    pm = _pair_mask(I, seed=5)
    pm[7, :] = False          # starting node: row 7 has no key at all
    pm[:, 11] = False         # ending node: column 11 has no key at all
    res, dtype = _run("evoformer_256", I, 0, pm)
    for node in NODES:
        assert_close(res[node], _want("evoformer_256", node, I, 0, pm), dtype, f"empty line {node}")
    assert np.all(res["start"][7] == 0.0) and np.all(res["end"][:, 11] == 0.0)


def test_residual_in_place_tensor_core_path():
    I, n_pad = 160, 10
    pm = _pair_mask(I, seed=6)
    res, dtype = _run("masked_768", I, n_pad, pm, in_place=True)
    for node in NODES:
        assert_close(res[node], _want("masked_768", node, I, n_pad, pm, residual=True), dtype, f"Z += out {node}")


def test_residual_out_of_place_and_no_pair_mask():
    I, n_pad = 130, 5
    res, dtype = _run("masked_768", I, n_pad, None, residual=True)
    for node in NODES:
        assert_close(res[node], _want("masked_768", node, I, n_pad, None, residual=True), dtype, f"Z + out {node}")


def test_pair_mask_and_residual_simt_path():
    I = 64
    pm = _pair_mask(I, seed=8)
    res, dtype = _run("tiny_f32", I, 0, pm, in_place=True)
    assert dtype == "f32"
    for node in NODES:
        assert_close(res[node], _want("tiny_f32", node, I, 0, pm, residual=True), dtype, f"simt {node}")
    pm72 = _pair_mask(72, seed=9)
    res, _ = _run("evoformer_256", 72, 0, pm72, force_simt=True)
    for node in NODES:
        assert_close(res[node], _want("evoformer_256", node, 72, 0, pm72), "bf16", f"simt bf16 {node}")
