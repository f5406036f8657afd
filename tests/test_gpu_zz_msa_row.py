"""MSA row-wise gated attention with pair bias (tri_attn_msa_forward) against the
fp64 oracle, through the C ABI on a GPU: f32 and bf16 storage, both kernel paths
(the tcgen05 path at the Evoformer shape, the CUDA-core path elsewhere or when
forced), ragged residue counts, padded rows and gaps in the MSA mask, key
chunks, the in-place residual, and sampled rows of the full Evoformer-shaped
workload."""
import numpy as np
import pytest

from oracle import msa_row_attention
from tests.gpu_cases import assert_close

pytestmark = pytest.mark.gpu


def _run(name, S=None, I=None, key_chunks=1, residual=False, in_place=False, force_simt=False, want_path=None,
         affine=False):
    import torch
    import protein_pair_representation_gate_b300 as pkg
    from synth import make_msa_inputs, with_affine_params
    from synth.device import msa_inputs_to_device
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    inp = make_msa_inputs(name, S=S, I=I)
    if affine:
        inp = with_affine_params(inp)
    wl = inp.workload
    t = msa_inputs_to_device(inp, "cuda")
    op = pkg.MSARowAttention(wl.c_z, wl.heads, wl.head_dim, wl.I, wl.dtype, key_chunks=key_chunks,
                             force_simt=force_simt)
    if want_path is not None:
        assert op.path(wl.c_m) == want_path
    if in_place:
        ms = t["Ms"].clone()
        op(ms, t["Z"], t, msa_mask=t["msa_mask"], out=ms, residual=True)
        out = ms
    else:
        out = op(t["Ms"], t["Z"], t, msa_mask=t["msa_mask"], residual=residual)
    assert op.ctx.status_sync() == 0
    return inp, out.float().cpu().numpy().astype(np.float64)


def _want(inp, rows=None, residual=False):
    a = inp.oracle_args()
    return msa_row_attention(a["Ms"], a["Z"], a["msa_mask"], rows=rows, residual=residual,
                             **{k: a[k] for k in ("w_q", "w_k", "w_v", "w_g", "w_b", "w_o", "ln_m_gamma",
                                                  "ln_m_beta", "ln_z_gamma", "ln_z_beta", "b_g", "b_o")})


def test_msa_f32():
    import protein_pair_representation_gate_b300 as pkg
    inp, got = _run("msa_tiny_f32", want_path=pkg.PATH_SIMT)
    assert_close(got, _want(inp), "f32", "msa f32")
    assert np.all(got[inp.msa_mask == 0] == 0.0)


@pytest.mark.parametrize("S, I", [(8, 72), (5, 130), (1, 1), (3, 300)])
def test_msa_bf16_evoformer_shape(S, I):
    """The tensor-core path: one query block (I <= 256) and two (I = 300), ragged."""
    import protein_pair_representation_gate_b300 as pkg
    inp, got = _run("msa_evoformer_512", S=S, I=I, want_path=pkg.PATH_SM103)
    assert_close(got, _want(inp), "bf16", f"msa bf16 S={S} I={I}")
    assert np.all(got[inp.msa_mask == 0] == 0.0)


def test_msa_bf16_simt_forced():
    import protein_pair_representation_gate_b300 as pkg
    inp, got = _run("msa_evoformer_512", S=4, I=72, force_simt=True, want_path=pkg.PATH_SIMT)
    assert_close(got, _want(inp), "bf16", "msa bf16 simt")
    assert np.all(got[inp.msa_mask == 0] == 0.0)


@pytest.mark.parametrize("force_simt", [False, True])
def test_msa_affine_params(force_simt):
    """Non-trivial LayerNorm gamma / beta on both sides, gate bias and output bias."""
    import protein_pair_representation_gate_b300 as pkg
    want_path = pkg.PATH_SIMT if force_simt else pkg.PATH_SM103
    inp, got = _run("msa_evoformer_512", S=5, I=130, force_simt=force_simt, want_path=want_path, affine=True)
    assert_close(got, _want(inp), "bf16", f"msa affine simt={force_simt}")
    assert np.all(got[inp.msa_mask == 0] == 0.0)
    inp, got = _run("msa_tiny_f32", affine=True)
    assert_close(got, _want(inp), "f32", "msa affine f32")


@pytest.mark.parametrize("S, I, chunks", [(6, 100, 3), (3, 300, 2)])
def test_msa_key_chunks(S, I, chunks):
    inp, got = _run("msa_evoformer_512", S=S, I=I, key_chunks=chunks)
    assert_close(got, _want(inp), "bf16", f"msa key chunks {chunks}")


def test_msa_residual_in_place_and_out_of_place():
    inp, got = _run("msa_tiny_f32", residual=True)
    assert_close(got, _want(inp, residual=True), "f32", "msa Ms + out")
    inp, got = _run("msa_evoformer_512", S=6, I=72, in_place=True)
    assert_close(got, _want(inp, residual=True), "bf16", "msa Ms += out")
    inp, got = _run("msa_evoformer_512", S=5, I=130, residual=True)
    assert_close(got, _want(inp, residual=True), "bf16", "msa Ms + out (out of place)")


def test_msa_full_size_sampled_rows():
    """The full msa_evoformer_512 workload (S = 512, I = 256), rows sampled for the
    oracle: the first, a middle one, the last valid row and the last (padding) row."""
    import protein_pair_representation_gate_b300 as pkg
    inp, got = _run("msa_evoformer_512", want_path=pkg.PATH_SM103)
    S = inp.workload.S
    rows = [0, 257, S - inp.workload.pad_rows - 1, S - 1]
    assert_close(got[rows], _want(inp, rows=rows), "bf16", "msa full size")
    assert np.all(got[S - inp.workload.pad_rows:] == 0.0)
    assert np.all(got[inp.msa_mask == 0] == 0.0)


def test_msa_large_layernorm_scale_is_reported():
    """The tensor-core MSA path keeps f16 intermediates: an MSA LayerNorm scale far
    beyond a trained model's pushes q, k, v out of range, which the status word
    reports (never silent NaN); the context works again at the normal scale."""
    import torch
    import protein_pair_representation_gate_b300 as pkg
    from synth import make_msa_inputs
    from synth.device import msa_inputs_to_device
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    inp = make_msa_inputs("msa_evoformer_512", S=4, I=72)
    wl = inp.workload
    t = msa_inputs_to_device(inp, "cuda")
    op = pkg.MSARowAttention(wl.c_z, wl.heads, wl.head_dim, wl.I, wl.dtype)
    assert op.path(wl.c_m) == pkg.PATH_SM103
    w = dict(t)
    w["ln_m_gamma"] = t["ln_m_gamma"] * 1e5
    op(t["Ms"], t["Z"], w, msa_mask=t["msa_mask"])
    assert op.ctx.status_sync() == pkg._binding.ERANGE
    out = op(t["Ms"], t["Z"], t, msa_mask=t["msa_mask"])
    assert op.ctx.status_sync() == 0
    assert bool(torch.isfinite(out.float()).all())


def test_msa_long_rows_sampled():
    """Longer MSA rows on the tensor-core path: I = 600 (three 256-query blocks,
    ten key tiles per head, a ragged tail), S = 24, rows sampled for the oracle."""
    import protein_pair_representation_gate_b300 as pkg
    inp, got = _run("msa_evoformer_512", S=24, I=600, want_path=pkg.PATH_SM103)
    rows = [0, 11, 23 - inp.workload.pad_rows, 23]
    assert_close(got[rows], _want(inp, rows=rows), "bf16", "msa I=600 sampled rows")
    assert np.all(got[inp.msa_mask == 0] == 0.0)
