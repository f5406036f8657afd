"""ctypes binding of libtriattn.so: argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; torch is
used here for device memory and streams (tensors are passed by data_ptr()).
The binding raises if the shared library is missing: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libtriattn.so")

OK, EINVAL, EUNSUPPORTED, ENOMEM, ECUDA, ETIMEOUT, ERANGE = range(7)
STARTING, ENDING = 0, 1
F32, BF16, TF32 = 0, 1, 2
DTYPES = {"f32": F32, "bf16": BF16, "tf32": TF32}
PATH_SIMT, PATH_SM103, PATH_SM103_TF32 = 0, 1, 2
NODES = {"start": STARTING, "end": ENDING, STARTING: STARTING, ENDING: ENDING}

EXPORTS = ("tri_attn_create", "tri_attn_destroy", "tri_attn_path", "tri_attn_workspace_bytes",
           "tri_attn_forward", "tri_attn_status_sync", "tri_attn_set_timing", "tri_attn_kernel_times",
           "tri_attn_status_string", "tri_attn_forward_static", "tri_attn_debug_inject", "tri_attn_forward_ex",
           "tri_attn_msa_workspace_bytes", "tri_attn_msa_forward", "tri_attn_static_status",
           "tri_attn_static_debug_inject", "tri_attn_msa_path")
FAULT_NONE, FAULT_SKIP_STAGE = 0, 1


class TriAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [("c_z", ctypes.c_int), ("heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("I_max", ctypes.c_int), ("dtype", ctypes.c_int), ("ln_eps", ctypes.c_float),
                ("key_chunks", ctypes.c_int), ("force_simt", ctypes.c_int)]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("ln_gamma", "ln_beta", "w_q", "w_k", "w_v", "w_g", "w_b", "b_g", "w_o", "b_o")]


class Options(ctypes.Structure):
    _fields_ = [("pair_mask", ctypes.c_void_p), ("residual", ctypes.c_int)]


class MsaWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("ln_m_gamma", "ln_m_beta", "w_q", "w_k", "w_v", "w_g", "b_g", "w_o", "b_o",
                 "ln_z_gamma", "ln_z_beta", "w_b")]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (once).  Raises FileNotFoundError if it was not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise FileNotFoundError(f"{path} is missing: build it with "
                                "`python -m protein_pair_representation_gate_b300.build`")
    lib = ctypes.CDLL(path)
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.tri_attn_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(vp)]
    lib.tri_attn_create.restype = i
    lib.tri_attn_destroy.argtypes = [vp]
    lib.tri_attn_destroy.restype = None
    lib.tri_attn_path.argtypes = [vp]
    lib.tri_attn_path.restype = i
    lib.tri_attn_workspace_bytes.argtypes = [vp, i]
    lib.tri_attn_workspace_bytes.restype = sz
    lib.tri_attn_forward.argtypes = [vp, i, i, vp, vp, ctypes.POINTER(Weights), vp, sz, vp, vp]
    lib.tri_attn_forward.restype = i
    lib.tri_attn_forward_ex.argtypes = [vp, i, i, vp, vp, ctypes.POINTER(Options), ctypes.POINTER(Weights), vp, sz,
                                        vp, vp]
    lib.tri_attn_forward_ex.restype = i
    lib.tri_attn_msa_path.argtypes = [vp, i]
    lib.tri_attn_msa_path.restype = i
    lib.tri_attn_msa_workspace_bytes.argtypes = [vp, i, i]
    lib.tri_attn_msa_workspace_bytes.restype = sz
    lib.tri_attn_msa_forward.argtypes = [vp, i, i, i, vp, vp, vp, ctypes.POINTER(MsaWeights), i, vp, sz, vp, vp]
    lib.tri_attn_msa_forward.restype = i
    lib.tri_attn_status_sync.argtypes = [vp, vp]
    lib.tri_attn_status_sync.restype = i
    lib.tri_attn_set_timing.argtypes = [vp, i]
    lib.tri_attn_set_timing.restype = i
    lib.tri_attn_kernel_times.argtypes = [vp, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float), i]
    lib.tri_attn_kernel_times.restype = i
    lib.tri_attn_forward_static.argtypes = [i, i, vp, vp, ctypes.POINTER(Weights), ctypes.c_float, vp, vp]
    lib.tri_attn_forward_static.restype = i
    lib.tri_attn_static_status.argtypes = [vp]
    lib.tri_attn_static_status.restype = i
    lib.tri_attn_static_debug_inject.argtypes = [i]
    lib.tri_attn_static_debug_inject.restype = i
    lib.tri_attn_debug_inject.argtypes = [vp, i]
    lib.tri_attn_debug_inject.restype = i
    lib.tri_attn_status_string.argtypes = [i]
    lib.tri_attn_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().tri_attn_status_string(status).decode()


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream_ptr(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


@dataclass
class TriAttnConfig:
    c_z: int
    heads: int
    head_dim: int
    I_max: int
    dtype: str = "bf16"          # "f32", "bf16" or "tf32" (fp32 storage, TF32 tensor-core arithmetic)
    ln_eps: float = 1e-5
    key_chunks: int = 1
    force_simt: bool = False

    def to_c(self) -> Config:
        return Config(self.c_z, self.heads, self.head_dim, self.I_max, DTYPES[self.dtype],
                      self.ln_eps, self.key_chunks, int(self.force_simt))


def forward_static(node, I: int, Z, mask, weights: dict, out, ln_eps: float = 1e-5, stream=None) -> int:
    """tri_attn_forward_static (no context, no workspace: library-owned device scratch); returns the status."""
    lib = load_library()
    w = Weights(*[_ptr(weights.get(n)) for n, _ in Weights._fields_])
    return lib.tri_attn_forward_static(NODES.get(node, node), I, _ptr(Z), _ptr(mask), ctypes.byref(w), ln_eps,
                                       _ptr(out), _stream_ptr(stream))


def static_status(stream=None) -> int:
    """tri_attn_static_status: synchronise the stream, read and clear the static path's status word."""
    return load_library().tri_attn_static_status(_stream_ptr(stream))


def static_debug_inject(fault: int) -> int:
    """tri_attn_static_debug_inject: the next forward_static runs with the stage-skip test hook."""
    return load_library().tri_attn_static_debug_inject(fault)


class TriAttn:
    """One library context (tri_attn_create / tri_attn_destroy)."""

    def __init__(self, cfg: TriAttnConfig):
        self.lib = load_library()
        self.cfg = cfg
        h = ctypes.c_void_p()
        st = self.lib.tri_attn_create(ctypes.byref(cfg.to_c()), ctypes.byref(h))
        if st != OK:
            raise TriAttnError(st, "tri_attn_create")
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            self.lib.tri_attn_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self) -> int:
        return self._h.value

    @property
    def path(self) -> int:
        return self.lib.tri_attn_path(self._h)

    def workspace_bytes(self, I: int) -> int:
        return int(self.lib.tri_attn_workspace_bytes(self._h, I))

    def forward(self, node, I: int, Z, mask, weights: dict, workspace, out, stream=None,
                workspace_bytes: int | None = None, pair_mask=None, residual: bool = False) -> int:
        """tri_attn_forward(_ex) on device tensors (or raw pointers); raises on a non-OK status."""
        st = self.forward_status(node, I, Z, mask, weights, workspace, out, stream, workspace_bytes,
                                 pair_mask=pair_mask, residual=residual)
        if st != OK:
            raise TriAttnError(st, "tri_attn_forward")
        return st

    def forward_status(self, node, I, Z, mask, weights, workspace, out, stream=None, workspace_bytes=None,
                       pair_mask=None, residual: bool = False) -> int:
        """tri_attn_forward, or tri_attn_forward_ex when a pair mask or the residual is asked for."""
        w = Weights(*[_ptr(weights.get(n)) for n, _ in Weights._fields_])
        if workspace_bytes is None:
            workspace_bytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else 0
        if pair_mask is None and not residual:
            return self.lib.tri_attn_forward(self._h, NODES.get(node, node), I, _ptr(Z), _ptr(mask), ctypes.byref(w),
                                             _ptr(workspace), workspace_bytes, _ptr(out), _stream_ptr(stream))
        opt = Options(_ptr(pair_mask), 1 if residual else 0)
        return self.lib.tri_attn_forward_ex(self._h, NODES.get(node, node), I, _ptr(Z), _ptr(mask), ctypes.byref(opt),
                                            ctypes.byref(w), _ptr(workspace), workspace_bytes, _ptr(out),
                                            _stream_ptr(stream))

    def msa_path(self, c_m: int) -> int:
        return self.lib.tri_attn_msa_path(self._h, c_m)

    def msa_workspace_bytes(self, S: int, I: int) -> int:
        return int(self.lib.tri_attn_msa_workspace_bytes(self._h, S, I))

    def msa_forward_status(self, S: int, I: int, c_m: int, msa, msa_mask, Z, weights: dict, workspace, out,
                           residual: bool = False, stream=None, workspace_bytes: int | None = None) -> int:
        """tri_attn_msa_forward on device tensors (or raw pointers); returns the status."""
        w = MsaWeights(*[_ptr(weights.get(n)) for n, _ in MsaWeights._fields_])
        if workspace_bytes is None:
            workspace_bytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else 0
        return self.lib.tri_attn_msa_forward(self._h, S, I, c_m, _ptr(msa), _ptr(msa_mask), _ptr(Z), ctypes.byref(w),
                                             1 if residual else 0, _ptr(workspace), workspace_bytes, _ptr(out),
                                             _stream_ptr(stream))

    def msa_forward(self, *args, **kw) -> int:
        st = self.msa_forward_status(*args, **kw)
        if st != OK:
            raise TriAttnError(st, "tri_attn_msa_forward")
        return st

    def status_sync(self, stream=None) -> int:
        return self.lib.tri_attn_status_sync(self._h, _stream_ptr(stream))

    def debug_inject(self, fault: int) -> int:
        """Test hook: in the next forward's attention kernel, the CTA that takes the first work item skips one load, so its bounded waits run out."""
        return self.lib.tri_attn_debug_inject(self._h, fault)

    def set_timing(self, on: bool) -> None:
        self.lib.tri_attn_set_timing(self._h, int(on))

    def kernel_times(self) -> list[tuple[str, float]]:
        cap = 8192
        names = (ctypes.c_char_p * cap)()
        ms = (ctypes.c_float * cap)()
        n = self.lib.tri_attn_kernel_times(self._h, names, ms, cap)
        if n < 0:
            return []
        return [(names[k].decode(), float(ms[k])) for k in range(min(n, cap))]
