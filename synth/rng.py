"""Counter-based SplitMix64 + Box-Muller normals (numpy, vectorised).

SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014): the n-th output from state s is mix64(s + (n+1)*G)
with G = 0x9E3779B97F4A7C15 and mix64 the variant-13 finaliser
(xor-shift 30, *0xBF58476D1CE4E5B9, xor-shift 27, *0x94D049BB133111EB,
xor-shift 31), all arithmetic mod 2**64.

Each (seed, stream) pair starts from its own state
kappa = mix64(mix64(seed) + stream*G), so element n of a stream is a pure
function of (seed, stream, n): any slice can be generated independently.

Uniforms: u_n = ((x_n >> 11) + 1) * 2**-53, in (0, 1].
Normals (Box & Muller 1958): element pair (2m, 2m+1) uses r = sqrt(-2 ln u_2m),
t = 2*pi*u_(2m+1); z_2m = r cos t, z_(2m+1) = r sin t.
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def mix64_scalar(z: int) -> int:
    """Same finaliser on a Python int (used for stream keys and tests)."""
    m = (1 << 64) - 1
    z &= m
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    return z ^ (z >> 31)


def stream_state(seed: int, stream: int) -> int:
    m = (1 << 64) - 1
    return mix64_scalar((mix64_scalar(seed) + stream * 0x9E3779B97F4A7C15) & m)


def splitmix64_outputs(state: int, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of the SplitMix64 sequence from `state`."""
    with np.errstate(over="ignore"):
        n = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
        return _mix64(np.uint64(state) + n * GAMMA)


def uniform01(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    x = splitmix64_outputs(stream_state(seed, stream), start, count)
    return ((x >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, stream: int, count: int, out: np.ndarray | None = None) -> np.ndarray:
    """`count` standard normals (float64) of one stream, element order 0..count-1."""
    if out is None:
        out = np.empty(count, dtype=np.float64)
    state = stream_state(seed, stream)
    npairs = (count + 1) // 2
    for p0 in range(0, npairs, _CHUNK):
        p1 = min(npairs, p0 + _CHUNK)
        x = splitmix64_outputs(state, 2 * p0, 2 * (p1 - p0))
        u = ((x >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * (2.0 ** -53)
        r = np.sqrt(-2.0 * np.log(u[0::2]))
        t = (2.0 * np.pi) * u[1::2]
        e0, e1 = 2 * p0, min(count, 2 * p1)
        seg = np.empty(2 * (p1 - p0), dtype=np.float64)
        seg[0::2] = r * np.cos(t)
        seg[1::2] = r * np.sin(t)
        out[e0:e1] = seg[: e1 - e0]
    return out
