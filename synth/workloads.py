"""The five synthetic workloads and their seeded inputs.

Shapes follow the pair-representation sizes the pages discuss (68 to ~2750
residues; the Evoformer core in bf16).  Distributions: Z ~ N(0, 1); every
projection matrix ~ N(0, 1/fan_in) (fan_in = c_z for the q/k/v/bias/gate
projections, H*d for the output projection); LayerNorm gamma = 1, beta = 0;
gate bias = 1; output bias = 0.  Stream numbers: Z=0, W_q=1, W_k=2, W_v=3,
W_b=4, W_g=5, W_o=6.

Weight layout: x @ W with W stored [in, out] row-major; head h owns output
channels h*d .. h*d+d-1 (head-major concatenation).

Casts to bf16 use round-to-nearest-even on the float32 value, done here with
integer bit operations so that both sides of a parity check receive the very
same bits.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .rng import normal

STREAM_Z, STREAM_WQ, STREAM_WK, STREAM_WV, STREAM_WB, STREAM_WG, STREAM_WO = range(7)


@dataclass(frozen=True)
class Workload:
    name: str
    I: int
    c_z: int
    heads: int
    head_dim: int
    dtype: str                 # "f32" or "bf16": storage type of Z, weights and out
    n_pad: int = 0             # trailing tokens marked invalid in the token mask
    bias_scale: float = 1.0    # multiplies the generated W_b (data, not a kernel flag)
    block_offset: float = 0.0  # added to every channel of Z[i, j] when i, j share a chain
    chain_len: int = 0         # chain length for block_offset
    nodes: tuple = ("start",)
    key_chunks: tuple = (1,)   # key-chunk counts to run (1 = unchunked)
    seed: int = 0

    @property
    def C(self) -> int:
        return self.heads * self.head_dim

    def attention_flops(self) -> float:
        """Counted work of one forward: 4 * I^3 * H * d (QK^T and PV)."""
        return 4.0 * float(self.I) ** 3 * self.heads * self.head_dim


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", I=64, c_z=32, heads=4, head_dim=8, dtype="f32"),
    "evoformer_256": Workload("evoformer_256", I=256, c_z=128, heads=4, head_dim=32, dtype="bf16",
                              nodes=("start", "end")),
    "masked_768": Workload("masked_768", I=768, c_z=128, heads=4, head_dim=32, dtype="bf16",
                           n_pad=77, bias_scale=4.0, nodes=("start", "end")),
    "complex_2048": Workload("complex_2048", I=2048, c_z=128, heads=4, head_dim=32, dtype="bf16",
                             block_offset=2.0, chain_len=256, nodes=("start", "end")),
    "single_chain_2752": Workload("single_chain_2752", I=2752, c_z=128, heads=4, head_dim=32, dtype="bf16",
                                  nodes=("start",), key_chunks=(1, 8)),
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest-even); returns uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return ((b + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_round(x: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(f32_to_bf16_bits(x))


@dataclass
class Inputs:
    """One workload's inputs.

    Storage arrays hold what the library receives: float32 arrays for the f32
    workloads, uint16 bf16 bit patterns for the bf16 ones.  `widen(name)`
    returns the exact stored values as float64 for the oracle.
    """
    workload: Workload
    Z: np.ndarray          # [I, I, c_z]
    mask: np.ndarray       # [I] uint8, 1 = valid token
    w_q: np.ndarray        # [c_z, H*d]
    w_k: np.ndarray
    w_v: np.ndarray
    w_g: np.ndarray
    w_b: np.ndarray        # [c_z, H]
    w_o: np.ndarray        # [H*d, c_z]
    ln_gamma: np.ndarray   # [c_z] float32
    ln_beta: np.ndarray    # [c_z] float32
    b_g: np.ndarray        # [H*d] float32
    b_o: np.ndarray        # [c_z] float32
    extra: dict = field(default_factory=dict)

    def widen(self, name: str) -> np.ndarray:
        a = getattr(self, name)
        if a.dtype == np.uint16:
            return bf16_bits_to_f32(a).astype(np.float64)
        return a.astype(np.float64)

    def oracle_args(self) -> dict:
        """Float64 copies of every tensor, keyed as the oracle takes them."""
        names = ["Z", "w_q", "w_k", "w_v", "w_g", "w_b", "w_o", "ln_gamma", "ln_beta", "b_g", "b_o"]
        d = {n: self.widen(n) for n in names}
        d["mask"] = self.mask.astype(bool)
        return d


def _store(x32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return f32_to_bf16_bits(x32)
    return np.ascontiguousarray(x32, dtype=np.float32)


def _weight(seed: int, stream: int, rows: int, cols: int, fan_in: int, scale: float = 1.0) -> np.ndarray:
    w = normal(seed, stream, rows * cols).reshape(rows, cols) * (scale / np.sqrt(fan_in))
    return w.astype(np.float32)


def make_pair_tensor(wl: Workload, threads: int | None = None) -> np.ndarray:
    """Z as float32 before the storage cast (N(0,1) plus the optional chain offset).

    Row blocks are generated on a thread pool (numpy releases the GIL); every
    element is a pure function of (seed, stream, index), so the result does
    not depend on the thread count.
    """
    from concurrent.futures import ThreadPoolExecutor
    import os

    I, c = wl.I, wl.c_z
    z = np.empty(I * I * c, dtype=np.float32)
    rows_per = max(1, (1 << 21) // (I * c))
    blocks = [(r0, min(I, r0 + rows_per)) for r0 in range(0, I, rows_per)]

    def fill(b):
        r0, r1 = b
        n = (r1 - r0) * I * c
        tmp = np.empty(n, dtype=np.float64)
        _normal_slice(wl.seed, STREAM_Z, r0 * I * c, n, tmp)
        z[r0 * I * c: r1 * I * c] = tmp

    nthreads = threads or min(32, os.cpu_count() or 1)
    if nthreads <= 1 or len(blocks) == 1:
        for b in blocks:
            fill(b)
    else:
        with ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(fill, blocks))
    z = z.reshape(I, I, c)
    if wl.block_offset != 0.0:
        chain = np.arange(I) // wl.chain_len
        same = chain[:, None] == chain[None, :]
        z[same] += np.float32(wl.block_offset)
    return z


def _normal_slice(seed: int, stream: int, start: int, count: int, out: np.ndarray) -> None:
    """Elements start .. start+count-1 of a normal stream (start must be even)."""
    assert start % 2 == 0
    from .rng import stream_state, splitmix64_outputs
    state = stream_state(seed, stream)
    npairs = (count + 1) // 2
    x = splitmix64_outputs(state, start, 2 * npairs)
    u = ((x >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * (2.0 ** -53)
    r = np.sqrt(-2.0 * np.log(u[0::2]))
    t = (2.0 * np.pi) * u[1::2]
    seg = np.empty(2 * npairs, dtype=np.float64)
    seg[0::2] = r * np.cos(t)
    seg[1::2] = r * np.sin(t)
    out[:count] = seg[:count]


def make_inputs(wl: Workload | str, I: int | None = None) -> Inputs:
    """Seeded inputs of a workload (optionally at another token count I)."""
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    if I is not None and I != wl.I:
        from dataclasses import replace
        wl = replace(wl, I=I, n_pad=min(wl.n_pad, I))
    c, H, d, C, s = wl.c_z, wl.heads, wl.head_dim, wl.C, wl.seed
    z32 = make_pair_tensor(wl)
    mask = np.ones(wl.I, dtype=np.uint8)
    if wl.n_pad:
        mask[wl.I - wl.n_pad:] = 0
    return Inputs(
        workload=wl,
        Z=_store(z32, wl.dtype),
        mask=mask,
        w_q=_store(_weight(s, STREAM_WQ, c, C, c), wl.dtype),
        w_k=_store(_weight(s, STREAM_WK, c, C, c), wl.dtype),
        w_v=_store(_weight(s, STREAM_WV, c, C, c), wl.dtype),
        w_g=_store(_weight(s, STREAM_WG, c, C, c), wl.dtype),
        w_b=_store(_weight(s, STREAM_WB, c, H, c, wl.bias_scale), wl.dtype),
        w_o=_store(_weight(s, STREAM_WO, C, c, C), wl.dtype),
        ln_gamma=np.ones(c, dtype=np.float32),
        ln_beta=np.zeros(c, dtype=np.float32),
        b_g=np.ones(C, dtype=np.float32),
        b_o=np.zeros(c, dtype=np.float32),
    )


# ---------------------------------------------------------------- MSA row attention
# Inputs of MSA row-wise attention with pair bias: an MSA representation
# Ms[S, I, c_m] ~ N(0, 1) (stream 10), a pair representation Z[I, I, c_z] ~ N(0, 1)
# (stream 11), the MSA-side projections ~ N(0, 1/c_m) (streams 1, 2, 3, 5), the
# pair-bias projection ~ N(0, 1/c_z) (stream 4), W_o ~ N(0, 1/(H d)) (stream 6);
# LayerNorm gamma = 1, beta = 0 on both sides, gate bias 1, output bias 0.  The
# MSA mask: the last `pad_rows` rows are padding (all 0), the last `n_pad`
# residues are padding in every row, and every other position is a gap (0)
# with probability `p_gap` (uniforms of stream 12).
STREAM_MSA, STREAM_MSA_Z, STREAM_MSA_MASK = 10, 11, 12


@dataclass(frozen=True)
class MsaWorkload:
    name: str
    S: int                     # MSA rows
    I: int                     # residues
    c_m: int
    c_z: int
    heads: int
    head_dim: int
    dtype: str
    n_pad: int = 0
    pad_rows: int = 0
    p_gap: float = 0.0
    seed: int = 0

    @property
    def C(self) -> int:
        return self.heads * self.head_dim

    def attention_flops(self) -> float:
        """Counted work of one forward: 4 * S * I^2 * H * d (QK^T and PV)."""
        return 4.0 * self.S * float(self.I) ** 2 * self.heads * self.head_dim


MSA_WORKLOADS = {
    "msa_tiny_f32": MsaWorkload("msa_tiny_f32", S=6, I=40, c_m=16, c_z=8, heads=2, head_dim=8, dtype="f32",
                                n_pad=3, pad_rows=1, p_gap=0.1),
    # Evoformer MSA stack shape: c_m = 256, c_z = 128, 8 heads of 32
    "msa_evoformer_512": MsaWorkload("msa_evoformer_512", S=512, I=256, c_m=256, c_z=128, heads=8, head_dim=32,
                                     dtype="bf16", n_pad=11, pad_rows=24, p_gap=0.1),
}


@dataclass
class MsaInputs:
    workload: MsaWorkload
    Ms: np.ndarray             # [S, I, c_m] storage
    Z: np.ndarray              # [I, I, c_z] storage
    msa_mask: np.ndarray       # [S, I] uint8
    w_q: np.ndarray            # [c_m, C]
    w_k: np.ndarray
    w_v: np.ndarray
    w_g: np.ndarray
    w_o: np.ndarray            # [C, c_m]
    w_b: np.ndarray            # [c_z, H]
    ln_m_gamma: np.ndarray
    ln_m_beta: np.ndarray
    ln_z_gamma: np.ndarray
    ln_z_beta: np.ndarray
    b_g: np.ndarray
    b_o: np.ndarray

    TENSORS = ("Ms", "Z", "w_q", "w_k", "w_v", "w_g", "w_o", "w_b", "ln_m_gamma", "ln_m_beta", "ln_z_gamma",
               "ln_z_beta", "b_g", "b_o")

    def widen(self, name: str) -> np.ndarray:
        a = getattr(self, name)
        if a.dtype == np.uint16:
            return bf16_bits_to_f32(a).astype(np.float64)
        return a.astype(np.float64)

    def oracle_args(self) -> dict:
        d = {n: self.widen(n) for n in self.TENSORS}
        d["msa_mask"] = self.msa_mask.astype(bool)
        return d


def make_msa_inputs(wl: MsaWorkload | str, S: int | None = None, I: int | None = None) -> MsaInputs:
    """Seeded inputs of an MSA workload (optionally with other S or I)."""
    from dataclasses import replace
    from .rng import uniform01
    if isinstance(wl, str):
        wl = MSA_WORKLOADS[wl]
    if S is not None or I is not None:
        S_, I_ = S or wl.S, I or wl.I
        wl = replace(wl, S=S_, I=I_, n_pad=min(wl.n_pad, I_ // 8), pad_rows=min(wl.pad_rows, S_ // 4))
    S, I, cm, cz, H, C, s = wl.S, wl.I, wl.c_m, wl.c_z, wl.heads, wl.C, wl.seed
    ms = normal(s, STREAM_MSA, S * I * cm).reshape(S, I, cm).astype(np.float32)
    z = normal(s, STREAM_MSA_Z, I * I * cz).reshape(I, I, cz).astype(np.float32)
    mask = (uniform01(s, STREAM_MSA_MASK, 0, S * I).reshape(S, I) >= wl.p_gap).astype(np.uint8)
    if wl.n_pad:
        mask[:, I - wl.n_pad:] = 0
    if wl.pad_rows:
        mask[S - wl.pad_rows:] = 0
    return MsaInputs(
        workload=wl,
        Ms=_store(ms, wl.dtype),
        Z=_store(z, wl.dtype),
        msa_mask=mask,
        w_q=_store(_weight(s, STREAM_WQ, cm, C, cm), wl.dtype),
        w_k=_store(_weight(s, STREAM_WK, cm, C, cm), wl.dtype),
        w_v=_store(_weight(s, STREAM_WV, cm, C, cm), wl.dtype),
        w_g=_store(_weight(s, STREAM_WG, cm, C, cm), wl.dtype),
        w_o=_store(_weight(s, STREAM_WO, C, cm, C), wl.dtype),
        w_b=_store(_weight(s, STREAM_WB, cz, H, cz), wl.dtype),
        ln_m_gamma=np.ones(cm, dtype=np.float32),
        ln_m_beta=np.zeros(cm, dtype=np.float32),
        ln_z_gamma=np.ones(cz, dtype=np.float32),
        ln_z_beta=np.zeros(cz, dtype=np.float32),
        b_g=np.ones(C, dtype=np.float32),
        b_o=np.zeros(cm, dtype=np.float32),
    )


# ---------------------------------------------------------------- affine parameters
# The default workloads keep LayerNorm gamma = 1, beta = 0, gate bias 1 and output
# bias 0.  with_affine_params swaps in seeded non-trivial values so that a test
# sees every term those parameters enter: gamma ~ 1 + 0.25 N(0, 1), beta, gate
# bias and output bias ~ 0.25 N(0, 1), each from its own stream (20 + its index
# in AFFINE_FIELDS).
AFFINE_FIELDS = ("ln_gamma", "ln_beta", "b_g", "b_o", "ln_m_gamma", "ln_m_beta", "ln_z_gamma", "ln_z_beta")
STREAM_AFFINE = 20


def with_affine_params(inp):
    """A copy of `inp` (Inputs or MsaInputs) with seeded non-trivial LayerNorm,
    gate-bias and output-bias parameters (float32, like the defaults)."""
    from dataclasses import fields, replace
    names = {f.name for f in fields(inp)}
    seed = inp.workload.seed
    new = {}
    for k, name in enumerate(AFFINE_FIELDS):
        if name not in names:
            continue
        n = getattr(inp, name).shape[0]
        x = 0.25 * normal(seed, STREAM_AFFINE + k, n)
        if name.endswith("gamma"):
            x = x + 1.0
        new[name] = x.astype(np.float32)
    return replace(inp, **new)
