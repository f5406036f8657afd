"""Small random problems for the oracle pins (seeded through the shared generator)."""
import numpy as np

from synth.rng import normal


def rand(seed: int, stream: int, *shape, scale: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    return normal(seed, stream, n).reshape(shape) * scale


def small_problem(I=9, c=8, H=2, d=4, seed=11, n_pad=0, bias_scale=1.0):
    """Float64 Z and weights of a small problem in the oracle's argument layout."""
    C = H * d
    p = dict(
        Z=rand(seed, 0, I, I, c),
        w_q=rand(seed, 1, c, C, scale=c ** -0.5),
        w_k=rand(seed, 2, c, C, scale=c ** -0.5),
        w_v=rand(seed, 3, c, C, scale=c ** -0.5),
        w_b=rand(seed, 4, c, H, scale=bias_scale * c ** -0.5),
        w_g=rand(seed, 5, c, C, scale=c ** -0.5),
        w_o=rand(seed, 6, C, c, scale=C ** -0.5),
        ln_gamma=1.0 + 0.1 * rand(seed, 7, c),
        ln_beta=0.1 * rand(seed, 8, c),
        b_g=rand(seed, 9, C),
        b_o=0.1 * rand(seed, 10, c),
    )
    mask = np.ones(I, dtype=bool)
    if n_pad:
        mask[I - n_pad:] = False
    p["mask"] = mask
    return p


WEIGHT_KEYS = ("w_q", "w_k", "w_v", "w_g", "w_b", "w_o", "ln_gamma", "ln_beta", "b_g", "b_o")


def weights(p):
    return {k: p[k] for k in WEIGHT_KEYS}
