"""The shared input generator: published SplitMix64 values, bf16 rounding, workload shapes."""
import numpy as np
import torch

from synth import WORKLOADS, bf16_bits_to_f32, f32_to_bf16_bits, make_inputs
from synth.rng import normal, splitmix64_outputs, uniform01
from synth.workloads import STREAM_Z, _normal_slice


def test_splitmix64_reference_outputs():
    """First outputs of SplitMix64 from state 0, as produced by the authors' reference code."""
    got = [int(x) for x in splitmix64_outputs(0, 0, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_uniform_range_and_normal_moments():
    u = uniform01(0, 1, 0, 1 << 16)
    assert u.min() > 0.0 and u.max() <= 1.0
    z = normal(5, 2, 1 << 20)
    assert abs(z.mean()) < 5e-3 and abs(z.std() - 1.0) < 5e-3
    # 4th moment of a standard normal is 3
    assert abs((z ** 4).mean() - 3.0) < 0.05


def test_stream_slices_are_consistent():
    full = normal(0, STREAM_Z, 1000)
    part = np.empty(200)
    _normal_slice(0, STREAM_Z, 400, 200, part)
    np.testing.assert_array_equal(part, full[400:600])


def test_bf16_rounding_matches_torch():
    x = np.concatenate([normal(0, 3, 4096).astype(np.float32) * 100,
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 0.0, -0.0, 65504.0], np.float32)])
    ours = f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(bf16_bits_to_f32(ours), torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_workload_inputs_shapes_and_recipe():
    inp = make_inputs("masked_768", I=40)
    wl = inp.workload
    assert inp.Z.shape == (40, 40, 128) and inp.Z.dtype == np.uint16
    assert inp.mask.sum() == 40 - 77 or inp.mask.sum() == 0  # 77 pads clipped to I
    inp = make_inputs("masked_768", I=100)
    assert inp.mask.sum() == 23 and np.all(inp.mask[23:] == 0)
    wb = bf16_bits_to_f32(inp.w_b)
    assert wb.shape == (128, 4)
    # bias projection amplified x4: std about 4/sqrt(128)
    assert 0.25 < wb.std() < 0.45
    assert wl.bias_scale == 4.0
    tiny = make_inputs("tiny_f32")
    assert tiny.Z.dtype == np.float32 and tiny.Z.shape == (64, 64, 32)
    assert np.all(tiny.b_g == 1.0) and np.all(tiny.ln_gamma == 1.0) and np.all(tiny.ln_beta == 0.0)


def test_block_diagonal_offset():
    inp = make_inputs("complex_2048", I=20)
    z = bf16_bits_to_f32(inp.Z)
    # chain length 256 > 20: every pair is in the same chain -> mean near +2
    assert abs(z.mean() - 2.0) < 0.05
    wl = WORKLOADS["complex_2048"]
    assert wl.chain_len == 256 and wl.block_offset == 2.0


def test_msa_inputs_shapes_and_mask_structure():
    from synth import make_msa_inputs
    inp = make_msa_inputs("msa_evoformer_512", S=16, I=72)
    wl = inp.workload
    assert inp.Ms.shape == (16, 72, 256) and inp.Ms.dtype == np.uint16
    assert inp.Z.shape == (72, 72, 128) and inp.w_b.shape == (128, 8) and inp.w_o.shape == (256, 256)
    m = inp.msa_mask
    assert m.shape == (16, 72) and m.dtype == np.uint8
    assert not m[16 - wl.pad_rows:].any() and not m[:, 72 - wl.n_pad:].any()
    gaps = 1.0 - m[:16 - wl.pad_rows, :72 - wl.n_pad].mean()
    assert 0.0 < gaps < 0.25
    again = make_msa_inputs("msa_evoformer_512", S=16, I=72)
    np.testing.assert_array_equal(again.Ms, inp.Ms)
    np.testing.assert_array_equal(again.msa_mask, inp.msa_mask)
