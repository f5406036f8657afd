"""B300-native gated triangle self-attention (starting and ending node), and
MSA row attention with pair bias.

The computation runs in libtriattn.so (hand-written CUDA for sm_103a, C ABI in
include/tri_attn.h); this package is its Python binding.  torch provides
device memory and streams only.
"""
from ._binding import (
    BF16, ENDING, F32, PATH_SIMT, PATH_SM103, PATH_SM103_TF32, STARTING, TF32, EXPORTS,
    TriAttn, TriAttnConfig, TriAttnError, load_library, status_string,
)

WEIGHT_NAMES = ("ln_gamma", "ln_beta", "w_q", "w_k", "w_v", "w_g", "w_b", "b_g", "w_o", "b_o")


class TriangleAttention:
    """A context plus a cached workspace: out = op(node, Z, mask, weights).

    Z, weights and mask are torch CUDA tensors laid out as tri_attn.h states
    (bf16 storage as torch.bfloat16 or raw int16 bits; fp32 storage for the
    "f32" and "tf32" dtypes).  Returns `out`.
    """

    def __init__(self, c_z: int, heads: int, head_dim: int, I_max: int, dtype: str = "bf16",
                 key_chunks: int = 1, ln_eps: float = 1e-5, force_simt: bool = False):
        self.ctx = TriAttn(TriAttnConfig(c_z, heads, head_dim, I_max, dtype, ln_eps, key_chunks, force_simt))
        self._ws = None

    @property
    def path(self) -> int:
        return self.ctx.path

    def workspace(self, I: int, device):
        import torch
        need = self.ctx.workspace_bytes(I)
        if self._ws is None or self._ws.numel() < need or self._ws.device != device:
            self._ws = None
            self._ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        return self._ws

    def __call__(self, node, Z, weights: dict, mask=None, out=None, stream=None, pair_mask=None,
                 residual: bool = False):
        """out = update (or Z + update with residual=True; pass out=Z for the in-place Z += update).
        pair_mask: optional [I, I] uint8 device tensor over the pairs of Z."""
        import torch
        I = Z.shape[0]
        if out is None:
            out = torch.empty_like(Z)
        ws = self.workspace(I, Z.device)
        self.ctx.forward(node, I, Z, mask, weights, ws, out, stream, pair_mask=pair_mask, residual=residual)
        return out


MSA_WEIGHT_NAMES = ("ln_m_gamma", "ln_m_beta", "w_q", "w_k", "w_v", "w_g", "b_g", "w_o", "b_o",
                    "ln_z_gamma", "ln_z_beta", "w_b")


class MSARowAttention:
    """MSA row-wise gated attention with pair bias: out = op(msa, Z, weights).

    msa [S, I, c_m] and Z [I, I, c_z] are torch CUDA tensors (tri_attn.h,
    tri_attn_msa_forward); weights holds MSA_WEIGHT_NAMES; msa_mask is an
    optional [S, I] uint8 tensor.  Returns `out` ([S, I, c_m]).
    """

    def __init__(self, c_z: int, heads: int, head_dim: int, I_max: int, dtype: str = "bf16",
                 key_chunks: int = 1, ln_eps: float = 1e-5, force_simt: bool = False):
        self.ctx = TriAttn(TriAttnConfig(c_z, heads, head_dim, I_max, dtype, ln_eps, key_chunks, force_simt))
        self._ws = None

    def path(self, c_m: int) -> int:
        """PATH_SM103 or PATH_SIMT: the kernels a forward with c_m MSA channels runs."""
        return self.ctx.msa_path(c_m)

    def workspace(self, S: int, I: int, device):
        import torch
        need = self.ctx.msa_workspace_bytes(S, I)
        if self._ws is None or self._ws.numel() < need or self._ws.device != device:
            self._ws = None
            self._ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        return self._ws

    def __call__(self, msa, Z, weights: dict, msa_mask=None, out=None, residual: bool = False, stream=None):
        """out = update (or msa + update with residual=True; out=msa updates in place)."""
        import torch
        S, I, c_m = msa.shape
        if out is None:
            out = torch.empty_like(msa)
        ws = self.workspace(S, I, msa.device)
        self.ctx.msa_forward(S, I, c_m, msa, msa_mask, Z, weights, ws, out, residual=residual, stream=stream)
        return out


__all__ = ["TriangleAttention", "MSARowAttention", "MSA_WEIGHT_NAMES", "TriAttn", "TriAttnConfig", "TriAttnError", "load_library", "status_string",
           "STARTING", "ENDING", "F32", "BF16", "TF32", "PATH_SIMT", "PATH_SM103", "PATH_SM103_TF32", "EXPORTS",
           "WEIGHT_NAMES"]
