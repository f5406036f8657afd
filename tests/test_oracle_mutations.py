"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin catches each.

The planted versions live only inside these tests, applied with monkeypatch;
the oracle module itself is never edited.
"""
import numpy as np
import pytest

import oracle.tri_attn_oracle as T
from tests import test_oracle_pins as pins


def _transposed_bias(Z, ln_gamma, ln_beta, w_b, block_rows=64):
    return _orig_pair_bias(Z, ln_gamma, ln_beta, w_b, block_rows).transpose(0, 2, 1).copy()


_orig_pair_bias = T.pair_bias
_orig_attention = T.softmax_attention
_orig_layer_norm = T.layer_norm


def _no_scale_attention(q, k, v, bias, key_valid):
    return _orig_attention(q * np.sqrt(q.shape[-1]), k, v, bias, key_valid)


def _unbiased_ln(x, gamma, beta, eps=T.LN_EPS):
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).sum(axis=-1, keepdims=True) / (x.shape[-1] - 1)
    return (x - mu) / np.sqrt(var + eps) * gamma + beta


def _unmasked_attention(q, k, v, bias, key_valid):
    return _orig_attention(q, k, v, bias, np.ones_like(key_valid))


def _gate_after_projection(o_heads, g, w_o, b_o):
    H, N, d = o_heads.shape
    u = o_heads.transpose(1, 0, 2).reshape(N, H * d)
    return u @ w_o + b_o


def _swapped_roles_ending(Z, mask, w_q, w_k, w_v, w_g, w_b, w_o, ln_gamma, ln_beta, b_g, b_o,
                          cols=None, key_chunks=1, bias=None, pair_mask=None):
    # keys/values taken along the row instead of down the column
    out = T.triangle_attention_starting(Z.transpose(1, 0, 2).copy(), mask, w_q, w_k, w_v, w_g, w_b, w_o,
                                        ln_gamma, ln_beta, b_g, b_o, key_chunks=key_chunks)
    return out


MUTATIONS = [
    ("pair bias transposed", "pair_bias", _transposed_bias,
     [lambda: pins.test_bias_orientation("start"), lambda: pins.test_bias_orientation("end")]),
    ("1/sqrt(d) dropped", "softmax_attention", _no_scale_attention,
     [lambda: pins.test_attention_core_matches_torch_sdpa(16, 33, 8, 5)]),
    ("unbiased variance in LayerNorm", "layer_norm", _unbiased_ln,
     [pins.test_layer_norm_matches_torch, pins.test_layer_norm_closed_form_moments]),
    ("key mask ignored", "softmax_attention", _unmasked_attention,
     [pins.test_single_valid_key_returns_its_value, pins.test_softmax_rows_sum_to_one_and_masked_keys_get_zero]),
    ("gate dropped", "_gate_and_project", _gate_after_projection,
     [lambda: pins.test_single_token_closed_form("start"), pins.test_gate_closed_out_gives_output_bias]),
    ("ending node reads Z untransposed", "triangle_attention_ending", _swapped_roles_ending,
     [pins.test_ending_equals_starting_on_transpose, lambda: pins.test_bias_orientation("end")]),
]


@pytest.mark.parametrize("name,attr,planted,checks", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pin_catches_planted_mistake(monkeypatch, name, attr, planted, checks):
    monkeypatch.setattr(T, attr, planted)
    for check in checks:
        with pytest.raises(AssertionError):
            check()
