"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test names the mistake it would catch.  Library special cases use torch
(fp64, CPU) and scipy; the rest are closed forms and invariants of the
operation.  No test here touches the CUDA library.
"""
import numpy as np
import pytest
import scipy.special
import torch

import oracle.tri_attn_oracle as O
from tests.oracle_cases import rand, small_problem, weights


def run(node, p, lines=None, key_chunks=1):
    return O.triangle_attention(node, p["Z"], p["mask"], weights(p), lines=lines, key_chunks=key_chunks)


# ---------------------------------------------------------------- LayerNorm

def test_layer_norm_matches_torch():
    """Library special case: torch.nn.functional.layer_norm (biased variance, eps 1e-5)."""
    x = rand(1, 0, 37, 16)
    g, b = 1.0 + 0.2 * rand(1, 1, 16), 0.3 * rand(1, 2, 16)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (16,), torch.from_numpy(g), torch.from_numpy(b), eps=1e-5)
    np.testing.assert_allclose(O.layer_norm(x, g, b), ref.numpy(), rtol=0, atol=1e-13)


def test_layer_norm_closed_form_moments():
    """gamma=1, beta=0: mean 0, variance var/(var+eps) (catches unbiased var, wrong eps)."""
    x = rand(2, 0, 5, 64) * 0.01  # small variance so eps matters
    y = O.layer_norm(x, np.ones(64), np.zeros(64))
    var = x.var(axis=-1)
    np.testing.assert_allclose(y.mean(axis=-1), 0.0, atol=1e-12)
    np.testing.assert_allclose(y.var(axis=-1), var / (var + 1e-5), rtol=1e-12)


def test_sigmoid_matches_scipy():
    x = rand(3, 0, 1000) * 10
    np.testing.assert_allclose(O.sigmoid(x), scipy.special.expit(x), rtol=1e-14, atol=0)


# ---------------------------------------------------------------- attention core

@pytest.mark.parametrize("nq,nk,d,npad", [(5, 7, 4, 0), (16, 33, 8, 5), (1, 1, 3, 0)])
def test_attention_core_matches_torch_sdpa(nq, nk, d, npad):
    """Library special case: SDPA(q, k, v, attn_mask = bias + -inf on invalid keys), fp64."""
    q, k, v = rand(4, 0, nq, d), rand(4, 1, nk, d), rand(4, 2, nk, 6)
    bias = rand(4, 3, nq, nk) * 2
    valid = np.ones(nk, dtype=bool)
    if npad:
        valid[-npad:] = False
    am = torch.from_numpy(np.where(valid[None, :], bias, -np.inf))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None], attn_mask=am[None])[0]
    np.testing.assert_allclose(O.softmax_attention(q, k, v, bias, valid), ref.numpy(), rtol=0, atol=1e-13)


def test_softmax_rows_sum_to_one_and_masked_keys_get_zero():
    """With V = identity the output is the probability matrix itself."""
    nk = 11
    q, k, bias = rand(5, 0, 6, 4), rand(5, 1, nk, 4), rand(5, 2, 6, nk) * 3
    valid = np.ones(nk, dtype=bool)
    valid[[2, 7, 10]] = False
    p = O.softmax_attention(q, k, np.eye(nk), bias, valid)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-14)
    assert np.all(p[:, ~valid] == 0.0)
    assert np.all(p[:, valid] > 0.0)


def test_zero_query_zero_bias_gives_mean_of_valid_values():
    nk = 9
    k, v = rand(6, 0, nk, 4), rand(6, 1, nk, 5)
    valid = np.array([1, 1, 0, 1, 0, 1, 1, 1, 0], dtype=bool)
    o = O.softmax_attention(np.zeros((3, 4)), k, v, np.zeros((3, nk)), valid)
    np.testing.assert_allclose(o, np.broadcast_to(v[valid].mean(axis=0), o.shape), atol=1e-14)


def test_single_valid_key_returns_its_value():
    nk = 6
    q, k, v, bias = rand(7, 0, 4, 3), rand(7, 1, nk, 3), rand(7, 2, nk, 2), rand(7, 3, 4, nk) * 5
    valid = np.zeros(nk, dtype=bool)
    valid[4] = True
    o = O.softmax_attention(q, k, v, bias, valid)
    np.testing.assert_array_equal(o, np.broadcast_to(v[4], o.shape))


def test_scale_applies_to_qk_only():
    """q.k / sqrt(d) + bias, not (q.k + bias) / sqrt(d): compare against SDPA with explicit scale."""
    d = 16
    q, k, v, bias = rand(8, 0, 3, d) * 3, rand(8, 1, 5, d) * 3, rand(8, 2, 5, 2), rand(8, 3, 3, 5) * 4
    valid = np.ones(5, dtype=bool)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None],
        attn_mask=torch.from_numpy(bias)[None], scale=1.0 / np.sqrt(d))[0]
    np.testing.assert_allclose(O.softmax_attention(q, k, v, bias, valid), ref.numpy(), atol=1e-13)


def test_joint_key_value_bias_permutation_invariance():
    nk = 13
    q, k, v, bias = rand(9, 0, 4, 4), rand(9, 1, nk, 4), rand(9, 2, nk, 3), rand(9, 3, 4, nk)
    valid = np.ones(nk, dtype=bool)
    valid[[0, 5]] = False
    perm = np.random.default_rng(0).permutation(nk)
    a = O.softmax_attention(q, k, v, bias, valid)
    b = O.softmax_attention(q, k[perm], v[perm], bias[:, perm], valid[perm])
    np.testing.assert_allclose(a, b, atol=1e-13)


@pytest.mark.parametrize("bounds", [
    [(0, 5), (5, 12), (12, 20)],
    [(0, 1), (1, 20)],
    [(0, 8), (8, 16), (16, 20)],
    [(0, 7), (7, 14), (14, 20)],
])
def test_chunked_lse_merge_equals_unchunked(bounds):
    """Key chunks merged by log-sum-exp equal one pass over all keys (incl. an all-masked chunk)."""
    nk = 20
    q, k, v, bias = rand(10, 0, 6, 4), rand(10, 1, nk, 4), rand(10, 2, nk, 5), rand(10, 3, 6, nk) * 4
    valid = np.ones(nk, dtype=bool)
    valid[8:16] = False  # the middle chunk of the third split has no valid key
    a = O.softmax_attention(q, k, v, bias, valid)
    b = O.chunked_softmax_attention(q, k, v, bias, valid, bounds)
    np.testing.assert_allclose(a, b, atol=1e-13)


# ---------------------------------------------------------------- whole operation

@pytest.mark.parametrize("node", ["start", "end"])
def test_single_token_closed_form(node):
    """I = 1: one key, p = 1, so out = (g * v) @ W_o + b_o with v, g from LN(Z[0,0])."""
    p = small_problem(I=1, c=8, H=2, d=3)
    zh = O.layer_norm(p["Z"][0, 0], p["ln_gamma"], p["ln_beta"])
    v = zh @ p["w_v"]
    g = scipy.special.expit(zh @ p["w_g"] + p["b_g"])
    want = (g * v) @ p["w_o"] + p["b_o"]
    np.testing.assert_allclose(run(node, p)[0, 0], want, atol=1e-13)


def test_gate_closed_out_gives_output_bias():
    """b_g -> -inf closes the gate: out = b_o on every valid pair (catches a missing gate)."""
    p = small_problem(I=6)
    p["b_g"] = np.full_like(p["b_g"], -1e3)
    for node in ("start", "end"):
        out = run(node, p)
        np.testing.assert_allclose(out, np.broadcast_to(p["b_o"], out.shape), atol=1e-12)


def test_ending_equals_starting_on_transpose():
    p = small_problem(I=10, n_pad=2)
    pt = dict(p, Z=p["Z"].transpose(1, 0, 2).copy())
    np.testing.assert_allclose(run("end", p), run("start", pt).transpose(1, 0, 2), atol=1e-13)


@pytest.mark.parametrize("node", ["start", "end"])
def test_token_permutation_equivariance(node):
    """out(P Z P^T, P m) = P out(Z) P^T (catches mixed-up row/column roles)."""
    p = small_problem(I=8, n_pad=1)
    perm = np.random.default_rng(3).permutation(8)
    pp = dict(p, Z=p["Z"][perm][:, perm].copy(), mask=p["mask"][perm])
    np.testing.assert_allclose(run(node, pp), run(node, p)[perm][:, perm], atol=1e-13)


@pytest.mark.parametrize("node", ["start", "end"])
def test_bias_orientation(node):
    """Scores from the bias alone, one dominant pair per query line.

    q = k = 0 (W_q = W_k = 0) and W_b reads one channel that is large on a
    chosen pair pattern only.  Starting node: query (i, j) must pick key
    k = pi(j) where Z[j, pi(j)] is marked (bias b[j, k]); ending node: query
    (i, j) must pick k = pi(i) where Z[pi(i), i] is marked (bias b[k, i]).
    A transposed bias picks pi^-1 instead.
    """
    I, c, H, d = 7, 16, 1, 4
    p = small_problem(I=I, c=c, H=H, d=d, seed=21)
    p["w_q"][:] = 0.0
    p["w_k"][:] = 0.0
    p["ln_gamma"][:] = 1.0
    p["ln_beta"][:] = 0.0
    pi = np.array([3, 0, 6, 1, 5, 2, 4])          # a permutation with no fixed point
    assert not np.array_equal(pi, np.argsort(pi))
    Z = p["Z"].copy()
    if node == "start":
        Z[np.arange(I), pi, 0] += 60.0             # pair (j, pi(j))
    else:
        Z[pi, np.arange(I), 0] += 60.0             # pair (pi(i), i)
    p["Z"] = Z
    p["w_b"][:] = 0.0
    p["w_b"][0, 0] = 20.0
    p["b_g"][:] = 1e3                              # gate fully open: g = 1
    p["b_o"][:] = 0.0
    wo_pinv = np.linalg.pinv(p["w_o"])             # recover u = o from out = o @ W_o
    out = run(node, p)
    o = out @ wo_pinv                              # [I, I, H*d]
    zh = O.layer_norm(Z, p["ln_gamma"], p["ln_beta"])
    v = zh @ p["w_v"]                              # v at every pair
    for i in range(I):
        for j in range(I):
            want = v[i, pi[j]] if node == "start" else v[pi[i], j]
            np.testing.assert_allclose(o[i, j], want, atol=1e-9)


@pytest.mark.parametrize("node", ["start", "end"])
def test_padded_pairs_have_no_influence(node):
    """Changing Z on any pair touching a padded token leaves every output unchanged."""
    p = small_problem(I=9, n_pad=3)
    base = run(node, p)
    Z = p["Z"].copy()
    pad = ~p["mask"]
    touched = pad[:, None] | pad[None, :]
    Z[touched] += rand(31, 0, int(touched.sum()), Z.shape[2]) * 5
    out = run(node, dict(p, Z=Z))
    np.testing.assert_allclose(out, base, atol=1e-13)
    assert np.all(out[touched] == 0.0)


@pytest.mark.parametrize("node", ["start", "end"])
def test_masked_equals_smaller_problem_zero_padded(node):
    """A problem with n trailing pads equals the unpadded (I - n) problem, zero-padded."""
    I, n = 12, 4
    p = small_problem(I=I, n_pad=n)
    small = dict(p, Z=p["Z"][: I - n, : I - n].copy(), mask=p["mask"][: I - n])
    big = run(node, p)
    np.testing.assert_allclose(big[: I - n, : I - n], run(node, small), atol=1e-13)
    assert np.all(big[I - n:] == 0.0) and np.all(big[:, I - n:] == 0.0)


def test_all_tokens_masked_gives_zero():
    p = small_problem(I=5)
    p["mask"][:] = False
    for node in ("start", "end"):
        out = run(node, p)
        assert np.all(out == 0.0) and np.all(np.isfinite(out))


@pytest.mark.parametrize("node", ["start", "end"])
@pytest.mark.parametrize("chunks", [2, 3, 5])
def test_whole_op_chunked_equals_unchunked(node, chunks):
    p = small_problem(I=11, n_pad=2)
    np.testing.assert_allclose(run(node, p, key_chunks=chunks), run(node, p), atol=1e-13)


@pytest.mark.parametrize("node", ["start", "end"])
def test_line_selection_matches_full(node):
    """Selecting output rows (start) / columns (end) returns the same values as the full run."""
    p = small_problem(I=10, n_pad=1)
    full = run(node, p)
    lines = [0, 3, 9, 4]
    part = run(node, p, lines=lines)
    if node == "start":
        np.testing.assert_array_equal(part, full[lines])
    else:
        np.testing.assert_array_equal(part, full[:, lines])


def test_brute_force_scalar_loops():
    """Independent scalar evaluation (math module, explicit loops) on a 3-token problem."""
    import math
    I, c, H, d = 3, 4, 2, 2
    p = small_problem(I=I, c=c, H=H, d=d, seed=41, n_pad=0)
    p["mask"][2] = False
    Z, m = p["Z"], p["mask"]

    def ln(x):
        mu = sum(x) / len(x)
        var = sum((t - mu) ** 2 for t in x) / len(x)
        return [(t - mu) / math.sqrt(var + 1e-5) * p["ln_gamma"][a] + p["ln_beta"][a] for a, t in enumerate(x)]

    def lin(x, w, col):
        return sum(x[a] * w[a][col] for a in range(len(x)))

    zh = [[ln(list(Z[a, b])) for b in range(I)] for a in range(I)]
    for node in ("start", "end"):
        out = run(node, p)
        for i in range(I):
            for j in range(I):
                if not (m[i] and m[j]):
                    assert all(out[i, j] == 0.0)
                    continue
                u = []
                for h in range(H):
                    qv = [lin(zh[i][j], p["w_q"], h * d + e) for e in range(d)]
                    scores, vals = [], []
                    for k in range(I):
                        if not m[k]:
                            continue
                        kp, bp = ((i, k), (j, k)) if node == "start" else ((k, j), (k, i))
                        kv = [lin(zh[kp[0]][kp[1]], p["w_k"], h * d + e) for e in range(d)]
                        s = sum(qv[e] * kv[e] for e in range(d)) / math.sqrt(d) + lin(zh[bp[0]][bp[1]], p["w_b"], h)
                        scores.append(s)
                        vals.append([lin(zh[kp[0]][kp[1]], p["w_v"], h * d + e) for e in range(d)])
                    mx = max(scores)
                    w = [math.exp(s - mx) for s in scores]
                    tot = sum(w)
                    for e in range(d):
                        g = 1.0 / (1.0 + math.exp(-(lin(zh[i][j], p["w_g"], h * d + e) + p["b_g"][h * d + e])))
                        u.append(g * sum(w[t] * vals[t][e] for t in range(len(w))) / tot)
                want = [sum(u[x] * p["w_o"][x][n] for x in range(H * d)) + p["b_o"][n] for n in range(c)]
                np.testing.assert_allclose(out[i, j], want, atol=1e-12)


# ---------------------------------------------------------------- pair mask and residual

def _pair_mask(I, seed, p_valid=0.7):
    rng = np.random.default_rng(seed)
    return rng.random((I, I)) < p_valid


def test_pair_mask_brute_force_scalar_loops():
    """Catches a pair mask applied to the wrong pair (transposed, or the query's
    instead of the key's): scalar loops on a 4-token problem, both nodes."""
    import math
    I, c, H, d = 4, 4, 2, 2
    p = small_problem(I=I, c=c, H=H, d=d, seed=43, n_pad=0)
    p["mask"][3] = False
    M = _pair_mask(I, 5)
    M[0, 1] = True
    Z, m = p["Z"], p["mask"]

    def ln(x):
        mu = sum(x) / len(x)
        var = sum((t - mu) ** 2 for t in x) / len(x)
        return [(t - mu) / math.sqrt(var + 1e-5) * p["ln_gamma"][a] + p["ln_beta"][a] for a, t in enumerate(x)]

    def lin(x, w, col):
        return sum(x[a] * w[a][col] for a in range(len(x)))

    zh = [[ln(list(Z[a, b])) for b in range(I)] for a in range(I)]
    for node in ("start", "end"):
        out = O.triangle_attention(node, Z, m, weights(p), pair_mask=M)
        for i in range(I):
            for j in range(I):
                if not (m[i] and m[j] and M[i, j]):
                    assert all(out[i, j] == 0.0)
                    continue
                u = []
                for h in range(H):
                    qv = [lin(zh[i][j], p["w_q"], h * d + e) for e in range(d)]
                    scores, vals = [], []
                    for k in range(I):
                        kp, bp = ((i, k), (j, k)) if node == "start" else ((k, j), (k, i))
                        if not (m[k] and M[kp[0], kp[1]]):
                            continue
                        kv = [lin(zh[kp[0]][kp[1]], p["w_k"], h * d + e) for e in range(d)]
                        s = sum(qv[e] * kv[e] for e in range(d)) / math.sqrt(d) + lin(zh[bp[0]][bp[1]], p["w_b"], h)
                        scores.append(s)
                        vals.append([lin(zh[kp[0]][kp[1]], p["w_v"], h * d + e) for e in range(d)])
                    mx = max(scores)
                    w = [math.exp(s - mx) for s in scores]
                    tot = sum(w)
                    for e in range(d):
                        g = 1.0 / (1.0 + math.exp(-(lin(zh[i][j], p["w_g"], h * d + e) + p["b_g"][h * d + e])))
                        u.append(g * sum(w[t] * vals[t][e] for t in range(len(w))) / tot)
                want = [sum(u[x] * p["w_o"][x][n] for x in range(H * d)) + p["b_o"][n] for n in range(c)]
                np.testing.assert_allclose(out[i, j], want, atol=1e-12)


def test_pair_mask_of_token_mask_equals_token_mask():
    """Catches a pair mask that changes anything beyond the token mask it encodes."""
    p = small_problem(I=9, n_pad=2, seed=17)
    M = np.outer(p["mask"], p["mask"])
    for node in ("start", "end"):
        np.testing.assert_allclose(O.triangle_attention(node, p["Z"], p["mask"], weights(p), pair_mask=M),
                                   run(node, p), atol=1e-13)


@pytest.mark.parametrize("node", ["start", "end"])
def test_masked_key_pair_has_no_influence_on_its_line(node):
    """Catches a masked key still entering the softmax: perturbing Z at a pair that
    is masked as a key leaves that line's outputs unchanged."""
    p = small_problem(I=8, seed=19)
    M = _pair_mask(8, 7, 0.8)
    line, key = 2, 5
    if node == "start":
        M[line, key] = False
    else:
        M[key, line] = False
    base = O.triangle_attention(node, p["Z"], p["mask"], weights(p), pair_mask=M)
    q = dict(p)
    q["Z"] = p["Z"].copy()
    if node == "start":
        q["Z"][line, key] += 3.0 * rand(23, 0, p["Z"].shape[-1])
    else:
        q["Z"][key, line] += 3.0 * rand(23, 0, p["Z"].shape[-1])
    pert = O.triangle_attention(node, q["Z"], q["mask"], weights(q), pair_mask=M)
    if node == "start":
        np.testing.assert_allclose(pert[line], base[line], atol=1e-12)
        assert not np.allclose(pert, base)               # the pair still feeds other lines' bias
    else:
        np.testing.assert_allclose(pert[:, line], base[:, line], atol=1e-12)
        assert not np.allclose(pert, base)


def test_residual_with_everything_masked_returns_z():
    """Catches a residual that scales or drops Z: with every pair masked the
    update is exactly 0, so the result is Z itself."""
    p = small_problem(I=6, seed=29)
    M = np.zeros((6, 6), dtype=bool)
    for node in ("start", "end"):
        got = O.triangle_attention(node, p["Z"], p["mask"], weights(p), pair_mask=M, residual=True)
        np.testing.assert_array_equal(got, p["Z"])
