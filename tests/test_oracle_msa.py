"""Pins of the oracle's MSA row attention with pair bias, each independent of the
function's own arithmetic: a reduction to the (separately pinned) starting-node
triangle attention, scalar loops on a tiny problem, and invariances that a
dropped term, a transposed bias or a mixed-up row would break."""
import math

import numpy as np
import pytest

import oracle.tri_attn_oracle as T
from tests.oracle_cases import rand


def msa_problem(S=5, I=7, c_m=8, c_z=6, H=2, d=4, seed=21, p_valid=0.75):
    C = H * d
    p = dict(
        Ms=rand(seed, 0, S, I, c_m),
        Z=rand(seed, 11, I, I, c_z),
        w_q=rand(seed, 1, c_m, C, scale=c_m ** -0.5),
        w_k=rand(seed, 2, c_m, C, scale=c_m ** -0.5),
        w_v=rand(seed, 3, c_m, C, scale=c_m ** -0.5),
        w_b=rand(seed, 4, c_z, H, scale=c_z ** -0.5),
        w_g=rand(seed, 5, c_m, C, scale=c_m ** -0.5),
        w_o=rand(seed, 6, C, c_m, scale=C ** -0.5),
        ln_m_gamma=1.0 + 0.1 * rand(seed, 7, c_m),
        ln_m_beta=0.1 * rand(seed, 8, c_m),
        ln_z_gamma=1.0 + 0.1 * rand(seed, 12, c_z),
        ln_z_beta=0.1 * rand(seed, 13, c_z),
        b_g=rand(seed, 9, C),
        b_o=0.1 * rand(seed, 10, c_m),
    )
    mask = np.random.default_rng(seed).random((S, I)) < p_valid
    mask[:, 0] = True                      # every row keeps a key
    return p, mask


def run(p, mask, **kw):
    return T.msa_row_attention(p["Ms"], p["Z"], mask, **{k: v for k, v in p.items() if k not in ("Ms", "Z")}, **kw)


def test_reduces_to_starting_node_triangle_attention():
    """With Ms = Z (S = I, one LayerNorm for both) the MSA row s is the starting
    node's row i = s, and the MSA mask is the pair mask."""
    p, mask = msa_problem(S=7, I=7, c_m=6, c_z=6)
    p["Ms"] = p["Z"].copy()
    p["ln_z_gamma"], p["ln_z_beta"] = p["ln_m_gamma"], p["ln_m_beta"]
    got = run(p, mask)
    tri = T.triangle_attention_starting(
        p["Z"], np.ones(7, dtype=bool), p["w_q"], p["w_k"], p["w_v"], p["w_g"], p["w_b"], p["w_o"],
        p["ln_m_gamma"], p["ln_m_beta"], p["b_g"], p["b_o"], pair_mask=mask)
    np.testing.assert_allclose(got, tri, rtol=0, atol=1e-12)


def _scalar_reference(p, mask):
    """The operation written out with scalar loops (no matrix routine)."""
    Ms, Z = p["Ms"], p["Z"]
    S, I, c_m = Ms.shape
    c_z = Z.shape[2]
    H = p["w_b"].shape[1]
    C = p["w_q"].shape[1]
    d = C // H

    def ln(vec, gamma, beta):
        n = len(vec)
        mu = sum(vec) / n
        var = sum((x - mu) ** 2 for x in vec) / n
        return [(vec[a] - mu) / math.sqrt(var + 1e-5) * gamma[a] + beta[a] for a in range(n)]

    def proj(vec, w, col):
        return sum(vec[a] * w[a][col] for a in range(len(vec)))

    bias = [[[0.0] * I for _ in range(I)] for _ in range(H)]
    for i in range(I):
        for j in range(I):
            zh = ln(list(Z[i, j]), p["ln_z_gamma"], p["ln_z_beta"])
            for h in range(H):
                bias[h][i][j] = proj(zh, p["w_b"], h)
    out = np.zeros((S, I, c_m))
    for s in range(S):
        mh = [ln(list(Ms[s, i]), p["ln_m_gamma"], p["ln_m_beta"]) for i in range(I)]
        q = [[proj(mh[i], p["w_q"], c) for c in range(C)] for i in range(I)]
        k = [[proj(mh[i], p["w_k"], c) for c in range(C)] for i in range(I)]
        v = [[proj(mh[i], p["w_v"], c) for c in range(C)] for i in range(I)]
        for i in range(I):
            if not mask[s, i]:
                continue
            u = [0.0] * C
            for h in range(H):
                sc = {}
                for j in range(I):
                    if mask[s, j]:
                        dot = sum(q[i][h * d + e] * k[j][h * d + e] for e in range(d))
                        sc[j] = dot / math.sqrt(d) + bias[h][i][j]
                top = max(sc.values())
                den = sum(math.exp(x - top) for x in sc.values())
                for e in range(d):
                    o = sum(math.exp(sc[j] - top) / den * v[j][h * d + e] for j in sc)
                    gate = 1.0 / (1.0 + math.exp(-(proj(mh[i], p["w_g"], h * d + e) + p["b_g"][h * d + e])))
                    u[h * d + e] = gate * o
            for c in range(c_m):
                out[s, i, c] = sum(u[a] * p["w_o"][a][c] for a in range(C)) + p["b_o"][c]
    return out


def test_scalar_loops_on_a_tiny_problem():
    p, mask = msa_problem(S=2, I=4, c_m=5, c_z=3, H=2, d=2, seed=5)
    mask[1, 2] = False
    np.testing.assert_allclose(run(p, mask), _scalar_reference(p, mask), rtol=0, atol=1e-12)


def test_rows_are_independent():
    p, mask = msa_problem()
    base = run(p, mask)
    p2 = dict(p, Ms=p["Ms"].copy())
    p2["Ms"][2] += 3.0 * rand(99, 0, *p["Ms"].shape[1:])
    moved = run(p2, mask)
    keep = [s for s in range(p["Ms"].shape[0]) if s != 2]
    np.testing.assert_array_equal(moved[keep], base[keep])
    assert np.abs(moved[2] - base[2]).max() > 1e-3


def test_pair_tensor_enters_only_through_the_bias():
    p, mask = msa_problem()
    p["w_b"] = np.zeros_like(p["w_b"])
    a = run(p, mask)
    p2 = dict(p, Z=rand(77, 0, *p["Z"].shape))
    np.testing.assert_array_equal(run(p2, mask), a)
    p3, _ = msa_problem()
    p4 = dict(p3, Z=rand(77, 0, *p3["Z"].shape))
    assert np.abs(run(p4, mask) - run(p3, mask)).max() > 1e-3


def test_row_permutation_equivariance():
    p, mask = msa_problem(S=6)
    perm = np.random.default_rng(1).permutation(6)
    base = run(p, mask)
    got = run(dict(p, Ms=p["Ms"][perm]), mask[perm])
    np.testing.assert_allclose(got, base[perm], rtol=0, atol=1e-12)


def test_residue_permutation_equivariance():
    """Relabelling residues (M's second axis, both axes of Z and the mask's
    residue axis) relabels the output: pins that M, Z and the mask index the
    same residues."""
    p, mask = msa_problem(I=8)
    perm = np.random.default_rng(2).permutation(8)
    base = run(p, mask)
    got = run(dict(p, Ms=p["Ms"][:, perm], Z=p["Z"][perm][:, perm]), mask[:, perm])
    np.testing.assert_allclose(got, base[:, perm], rtol=0, atol=1e-12)


def test_bias_orientation_query_by_key():
    """A dominant bias on pair (i0, j0) of Z makes query i0 of every row copy
    the value at key j0 (and not query j0 the value at key i0)."""
    p, mask = msa_problem(S=3, I=6, p_valid=1.0)
    i0, j0 = 1, 4
    p["w_b"] = np.zeros_like(p["w_b"])
    p["w_b"][0, :] = 1.0
    p["ln_z_beta"] = np.zeros_like(p["ln_z_beta"])
    p["ln_z_gamma"] = np.ones_like(p["ln_z_gamma"])
    p["Z"] = np.zeros_like(p["Z"])
    p["Z"][:, :, 1] = 1.0                  # every pair normalises to the same vector ...
    p["Z"][i0, j0] = 0.0
    p["Z"][i0, j0, 0] = 1.0                # ... except (i0, j0), whose channel 0 is large after LN
    b = T.pair_bias(p["Z"], p["ln_z_gamma"], p["ln_z_beta"], p["w_b"])
    assert b[0, i0, j0] > b[0, i0, j0 - 1] + 2.0
    p["w_b"] *= 40.0                       # the bias then dominates every score of query i0
    p["w_q"] = np.zeros_like(p["w_q"])
    out = run(p, mask)
    mh = T.layer_norm(p["Ms"], p["ln_m_gamma"], p["ln_m_beta"])
    for s in range(3):
        v = mh[s] @ p["w_v"]
        g = T.sigmoid(mh[s, i0] @ p["w_g"] + p["b_g"])
        want = (g * v[j0]) @ p["w_o"] + p["b_o"]
        np.testing.assert_allclose(out[s, i0], want, rtol=0, atol=1e-9)
        g0 = T.sigmoid(mh[s, j0] @ p["w_g"] + p["b_g"])
        assert np.abs(out[s, j0] - ((g0 * v[i0]) @ p["w_o"] + p["b_o"])).max() > 1e-3


def test_masked_positions_and_masked_keys():
    p, mask = msa_problem()
    out = run(p, mask)
    assert np.all(out[~mask] == 0.0)
    # the values at a masked key have no influence on the row
    s, j = np.argwhere(~mask)[0]
    p2 = dict(p, Ms=p["Ms"].copy())
    p2["Ms"][s, j] += 5.0
    np.testing.assert_array_equal(run(p2, mask), out)
    # a fully masked row is 0; with the residual it is the row itself
    mask2 = mask.copy()
    mask2[3] = False
    np.testing.assert_array_equal(run(p, mask2)[3], 0.0)
    np.testing.assert_array_equal(run(p, mask2, residual=True)[3], p["Ms"][3])


def test_residual_adds_the_input():
    p, mask = msa_problem()
    np.testing.assert_allclose(run(p, mask, residual=True), p["Ms"] + run(p, mask), rtol=0, atol=1e-15)


def test_single_valid_key_returns_its_gated_value():
    p, mask = msa_problem(S=2, I=5)
    mask[:] = False
    mask[:, 3] = True
    out = run(p, mask)
    mh = T.layer_norm(p["Ms"], p["ln_m_gamma"], p["ln_m_beta"])
    for s in range(2):
        g = T.sigmoid(mh[s, 3] @ p["w_g"] + p["b_g"])
        want = (g * (mh[s, 3] @ p["w_v"])) @ p["w_o"] + p["b_o"]
        np.testing.assert_allclose(out[s, 3], want, rtol=0, atol=1e-12)


@pytest.mark.parametrize("planted", ["bias transposed", "MSA LayerNorm affine dropped"])
def test_pins_catch_planted_mistakes(monkeypatch, planted):
    orig_bias = T.pair_bias
    orig_msa = T.msa_row_attention
    if planted == "bias transposed":
        monkeypatch.setattr(T, "pair_bias",
                            lambda Z, g, b, w, block_rows=64: orig_bias(Z, g, b, w, block_rows).transpose(0, 2, 1).copy())
        checks = [test_scalar_loops_on_a_tiny_problem, test_bias_orientation_query_by_key]
    else:
        def wrong(Ms, Z, msa_mask, w_q, w_k, w_v, w_g, w_b, w_o, ln_m_gamma, ln_m_beta, ln_z_gamma, ln_z_beta,
                  b_g, b_o, rows=None, bias=None, residual=False):
            return orig_msa(Ms, Z, msa_mask, w_q, w_k, w_v, w_g, w_b, w_o, np.ones_like(ln_m_gamma),
                            np.zeros_like(ln_m_beta), ln_z_gamma, ln_z_beta, b_g, b_o, rows=rows, bias=bias,
                            residual=residual)
        monkeypatch.setattr(T, "msa_row_attention", wrong)
        checks = [test_scalar_loops_on_a_tiny_problem]
    for check in checks:
        with pytest.raises(AssertionError):
            check()
