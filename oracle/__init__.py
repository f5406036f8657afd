"""Plain fp64 CPU oracle for gated triangle self-attention (and MSA row attention
with pair bias).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this package: only the tests, the smoke check and the bench's CPU
baseline use it.  It shares no code with the CUDA library.
"""
from .tri_attn_oracle import (
    layer_norm,
    sigmoid,
    pair_bias,
    softmax_attention,
    chunked_softmax_attention,
    triangle_attention_starting,
    triangle_attention_ending,
    triangle_attention,
    msa_row_attention,
)

__all__ = [
    "layer_norm", "sigmoid", "pair_bias", "softmax_attention", "chunked_softmax_attention",
    "triangle_attention_starting", "triangle_attention_ending", "triangle_attention",
    "msa_row_attention",
]
