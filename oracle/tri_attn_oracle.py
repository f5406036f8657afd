"""fp64 oracle: pair-biased, gated triangle self-attention (starting and ending node).

TEST INFRASTRUCTURE ONLY -- the product path never imports this module.

What is computed (the operation the library implements):

  for a pair representation Z[I, I, c] and a per-token validity mask m[I],
    zh      = LayerNorm(Z)                      (per pair vector, biased variance, eps 1e-5)
    q, k, v = zh @ W_q, zh @ W_k, zh @ W_v      (H heads x d channels, no bias)
    g       = sigmoid(zh @ W_g + b_g)           (H*d channels)
    b[h]    = zh @ W_b[:, h]                    (one pair bias per head)
  starting node, row i, head h, query j, keys k with m[k] = 1:
    s_jk    = q[i,j,h] . k[i,k,h] / sqrt(d) + b[h, j, k]
    o[i,j,h]= sum_k softmax_k(s_jk) v[i,k,h]
  ending node (queries down column j, bias transposed):
    s_ik    = q[i,j,h] . k[k,j,h] / sqrt(d) + b[h, k, i]
    o[i,j,h]= sum_k softmax_k(s_ik) v[k,j,h]
  both:
    out[i,j]= (g[i,j] * concat_h o[i,j,h]) @ W_o + b_o,  and 0 where m[i]*m[j] = 0.
  optional pair mask M[I, I] (the Evoformer's use; a reading, the pages give no
  formula): the starting node's row i attends only keys (i, k) with M[i, k] = 1
  and its output pairs (i, j) with M[i, j] = 0 are 0; the ending node's column j
  attends keys (k, j) with M[k, j] = 1 and zeroes pairs (i, j) with M[i, j] = 0.
  optional residual: the result is Z + out (the in-place update Z += out).

  MSA row-wise gated self-attention with pair bias (the same attention with
  another batch and bias source): for an MSA representation Ms[S, I, c_m], a
  pair representation Z[I, I, c_z] and a mask mm[S, I],
    mh      = LayerNorm_m(Ms);  q, k, v, g from mh as above
    b[h]    = LayerNorm_z(Z) @ W_b[:, h]          (shared by all S rows)
  row s, head h, query i, keys j with mm[s, j] = 1:
    o[s,i,h]= sum_j softmax_j(q[s,i,h] . k[s,j,h] / sqrt(d) + b[h, i, j]) v[s,j,h]
    out[s,i]= (g[s,i] * concat_h o[s,i,h]) @ W_o + b_o, and 0 where mm[s, i] = 0.

Sources on the pages (none prints the formulas; these name the parts):
  * Dell, "PowerEdge XE8545 ... protein model analysis": the Evoformer handles
    the residue-pair graph with triangle self-attention (Evoformer paragraph).
  * Intel, "AlphaFold2 end-to-end optimisation on Xeon", step 2 (DL inference)
    and step 4: self-attention learns triangle-geometry constraints over the
    pair representation; the attention module carries a large bias term
    computed by tensor contractions from the pair tensor.
  * Intel, step 4 (the attention-slicing example): the attention call takes
    the query rows, a per-row (batched) mask bias and one bias shared by all
    rows (non-batched, from the pair representation) -- the MSA row form.
  * OpenFold-TRT summary (gist.science), Methodology: bf16 Evoformer core.
  * Design-CP summary (gist.science), Methodology 1: keys/values processed in
    pieces with scores formed on the fly (ring attention), self-attention
    recast as cross-attention over key shards -- the chunked form below.

Readings where the pages are silent (each also listed in the design notes):
  LayerNorm eps 1e-5 with biased variance; no bias on the q/k/v/pair-bias
  projections; gate bias and output bias present; the 1/sqrt(d) scale applies
  to q.k only; masked keys get -inf; output pairs touching a padded token are
  exactly 0 (so a fully masked row is 0, never NaN); the caller adds the
  residual.  Weights are stored [in, out]; head h owns channels h*d..h*d+d-1.

Parity pins live in tests/test_oracle_*.py (library special cases, closed
forms and invariants); every function here has at least one.
"""
from __future__ import annotations

import numpy as np

LN_EPS = 1e-5


def layer_norm(x: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float = LN_EPS) -> np.ndarray:
    """LayerNorm over the last axis: (x - mean) / sqrt(biased var + eps) * gamma + beta."""
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * gamma + beta


def sigmoid(x: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):          # exp(-x) -> inf gives the correct limit 0
        return 1.0 / (1.0 + np.exp(-x))


def pair_bias(Z: np.ndarray, ln_gamma, ln_beta, w_b, block_rows: int = 64) -> np.ndarray:
    """b[h, a, c] = LayerNorm(Z[a, c]) @ W_b[:, h] for every pair (a, c).

    The per-head attention bias derived from the pair tensor (Intel page, step 4:
    the bias term of the attention module, formed by tensor contractions).
    Computed in row blocks to bound fp64 temporaries.  Returns [H, I, I].
    """
    I = Z.shape[0]
    H = w_b.shape[1]
    out = np.empty((H, I, I), dtype=np.float64)
    for a0 in range(0, I, block_rows):
        a1 = min(I, a0 + block_rows)
        zh = layer_norm(Z[a0:a1], ln_gamma, ln_beta)           # [rows, I, c]
        out[:, a0:a1, :] = np.moveaxis(zh @ w_b, -1, 0)        # [H, rows, I]
    return out


def softmax_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, bias: np.ndarray,
                      key_valid: np.ndarray) -> np.ndarray:
    """One head of biased attention, two passes over a materialised score matrix.

    q [Nq, d], k [Nk, d], v [Nk, dv], bias [Nq, Nk], key_valid [Nk] bool.
    s = q k^T / sqrt(d) + bias, -inf on invalid keys; p = exp(s - max) / sum;
    returns p @ v.  A query whose keys are all invalid returns 0 (the caller
    zeroes such outputs anyway).
    """
    d = q.shape[-1]
    s = q @ k.T / np.sqrt(d) + bias
    s = np.where(key_valid[None, :], s, -np.inf)
    smax = s.max(axis=-1, keepdims=True)
    finite = np.isfinite(smax)
    e = np.exp(s - np.where(finite, smax, 0.0))
    denom = e.sum(axis=-1, keepdims=True)
    p = np.divide(e, denom, out=np.zeros_like(e), where=denom > 0)
    return p @ v


def chunked_softmax_attention(q, k, v, bias, key_valid, bounds) -> np.ndarray:
    """The same attention with keys split into chunks merged by log-sum-exp.

    Each chunk [c0, c1) yields a normalised partial o_c and lse_c =
    log sum_k exp(s_k) over its keys; the merged result is
    sum_c exp(lse_c - lse) o_c with lse = log sum_c exp(lse_c).  This is the
    cross-attention-over-key-shards / ring form of the Design-CP summary
    (Methodology 1), here on one machine.  Chunks with no valid key carry
    lse_c = -inf and weight 0.
    """
    d = q.shape[-1]
    nq = q.shape[0]
    parts, lses = [], []
    for c0, c1 in bounds:
        s = q @ k[c0:c1].T / np.sqrt(d) + bias[:, c0:c1]
        s = np.where(key_valid[None, c0:c1], s, -np.inf)
        m = s.max(axis=-1, keepdims=True) if c1 > c0 else np.full((nq, 1), -np.inf)
        finite = np.isfinite(m)
        e = np.exp(s - np.where(finite, m, 0.0))
        l = e.sum(axis=-1, keepdims=True)
        o = np.divide(e @ v[c0:c1], l, out=np.zeros((nq, v.shape[1])), where=l > 0)
        with np.errstate(divide="ignore"):
            lse = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
        parts.append(o)
        lses.append(lse)
    L = np.concatenate(lses, axis=1)                          # [nq, chunks]
    top = L.max(axis=1, keepdims=True)
    top_f = np.where(np.isfinite(top), top, 0.0)
    w = np.exp(L - top_f)                                     # exp(-inf) = 0 for empty chunks
    tot = w.sum(axis=1, keepdims=True)
    w = np.divide(w, tot, out=np.zeros_like(w), where=tot > 0)
    return sum(w[:, c:c + 1] * parts[c] for c in range(len(parts)))


def _chunk_bounds(n: int, chunks: int) -> list[tuple[int, int]]:
    if chunks <= 1:
        return [(0, n)]
    size = -(-n // chunks)
    return [(c0, min(n, c0 + size)) for c0 in range(0, n, size)]


def _heads(x: np.ndarray, H: int) -> np.ndarray:
    """[N, H*d] -> [H, N, d] (head h owns channels h*d .. h*d+d-1)."""
    N, C = x.shape
    return x.reshape(N, H, C // H).transpose(1, 0, 2)


def _gate_and_project(o_heads: np.ndarray, g: np.ndarray, w_o, b_o) -> np.ndarray:
    """(g * concat_h o_h) @ W_o + b_o for one line of pairs; o_heads [H, N, d]."""
    H, N, d = o_heads.shape
    u = g * o_heads.transpose(1, 0, 2).reshape(N, H * d)
    return u @ w_o + b_o


def triangle_attention_starting(Z, mask, w_q, w_k, w_v, w_g, w_b, w_o, ln_gamma, ln_beta, b_g, b_o,
                                rows=None, key_chunks: int = 1, bias=None, pair_mask=None) -> np.ndarray:
    """Starting-node triangle attention; returns out[rows, I, c] (all rows by default).

    Row i: queries are pairs (i, j), keys/values pairs (i, k), bias b[h, j, k].
    With a pair mask M, row i's keys and output pairs are further limited to
    M[i, :] = 1.
    """
    I, _, c = Z.shape
    H = w_b.shape[1]
    mask = np.asarray(mask, dtype=bool)
    rows = range(I) if rows is None else rows
    if bias is None:
        bias = pair_bias(Z, ln_gamma, ln_beta, w_b)
    bounds = _chunk_bounds(I, key_chunks)
    out = np.zeros((len(rows), I, c), dtype=np.float64)
    for r, i in enumerate(rows):
        if not mask[i]:
            continue
        valid = mask if pair_mask is None else mask & np.asarray(pair_mask[i], dtype=bool)
        zh = layer_norm(Z[i], ln_gamma, ln_beta)                # [I, c]
        q, k, v = _heads(zh @ w_q, H), _heads(zh @ w_k, H), _heads(zh @ w_v, H)
        g = sigmoid(zh @ w_g + b_g)
        o = np.empty_like(q)
        for h in range(H):
            if key_chunks <= 1:
                o[h] = softmax_attention(q[h], k[h], v[h], bias[h], valid)
            else:
                o[h] = chunked_softmax_attention(q[h], k[h], v[h], bias[h], valid, bounds)
        out[r] = _gate_and_project(o, g, w_o, b_o)
        out[r][~valid] = 0.0
    return out


def triangle_attention_ending(Z, mask, w_q, w_k, w_v, w_g, w_b, w_o, ln_gamma, ln_beta, b_g, b_o,
                              cols=None, key_chunks: int = 1, bias=None, pair_mask=None) -> np.ndarray:
    """Ending-node triangle attention; returns out[:, cols, c] as [I, len(cols), c].

    Column j: queries are pairs (i, j), keys/values pairs (k, j), bias b[h, k, i]
    (the pair bias read transposed).  Written directly, not by transposing Z, so
    that the identity end(Z) = start(Z^T)^T is a check rather than a definition.
    With a pair mask M, column j's keys and output pairs are further limited to
    M[:, j] = 1.
    """
    I, _, c = Z.shape
    H = w_b.shape[1]
    mask = np.asarray(mask, dtype=bool)
    cols = range(I) if cols is None else cols
    if bias is None:
        bias = pair_bias(Z, ln_gamma, ln_beta, w_b)
    bounds = _chunk_bounds(I, key_chunks)
    out = np.zeros((I, len(cols), c), dtype=np.float64)
    for r, j in enumerate(cols):
        if not mask[j]:
            continue
        valid = mask if pair_mask is None else mask & np.asarray(pair_mask[:, j], dtype=bool)
        zh = layer_norm(Z[:, j], ln_gamma, ln_beta)             # pairs (x, j), x = 0..I-1
        q, k, v = _heads(zh @ w_q, H), _heads(zh @ w_k, H), _heads(zh @ w_v, H)
        g = sigmoid(zh @ w_g + b_g)
        o = np.empty_like(q)
        for h in range(H):
            bt = bias[h].T                                      # bt[i, k] = b[h, k, i]
            if key_chunks <= 1:
                o[h] = softmax_attention(q[h], k[h], v[h], bt, valid)
            else:
                o[h] = chunked_softmax_attention(q[h], k[h], v[h], bt, valid, bounds)
        col = _gate_and_project(o, g, w_o, b_o)                 # [I (i), c]
        col[~valid] = 0.0
        out[:, r] = col
    return out


def triangle_attention(node: str, Z, mask, weights: dict, lines=None, key_chunks: int = 1, bias=None,
                       pair_mask=None, residual: bool = False):
    """Dispatch by node.  `lines` selects output rows (start) or columns (end).

    Returns out for the selected lines in the orientation of Z:
    start -> [len(lines), I, c]; end -> [I, len(lines), c].  With residual=True
    it returns Z + out over the same pairs.
    """
    w = {k: weights[k] for k in ("w_q", "w_k", "w_v", "w_g", "w_b", "w_o", "ln_gamma", "ln_beta", "b_g", "b_o")}
    sel = range(Z.shape[0]) if lines is None else list(lines)
    if node == "start":
        out = triangle_attention_starting(Z, mask, rows=lines, key_chunks=key_chunks, bias=bias,
                                          pair_mask=pair_mask, **w)
        return Z[sel] + out if residual else out
    if node == "end":
        out = triangle_attention_ending(Z, mask, cols=lines, key_chunks=key_chunks, bias=bias,
                                        pair_mask=pair_mask, **w)
        return Z[:, sel] + out if residual else out
    raise ValueError(f"node must be 'start' or 'end', got {node!r}")


def msa_row_attention(Ms, Z, msa_mask, w_q, w_k, w_v, w_g, w_b, w_o, ln_m_gamma, ln_m_beta, ln_z_gamma,
                      ln_z_beta, b_g, b_o, rows=None, bias=None, residual: bool = False) -> np.ndarray:
    """MSA row-wise gated self-attention with pair bias; returns [len(rows), I, c_m].

    Row s of the MSA representation Ms[S, I, c_m] attends over its own residues:
    queries (s, i), keys/values (s, j) with msa_mask[s, j] = 1, and the per-head
    bias b[h, i, j] = LayerNorm_z(Z[i, j]) @ W_b[:, h] from the pair
    representation, the same for every row (the non-batched bias of the Intel
    page's attention call, step 4; the per-row mask is its batched bias).  The
    MSA and the pair tensor have LayerNorms of their own.  Outputs at masked
    positions (s, i) are 0; with residual=True the result is Ms + out.
    """
    S, I, _ = Ms.shape
    H = w_b.shape[1]
    msa_mask = np.asarray(msa_mask, dtype=bool)
    rows = range(S) if rows is None else rows
    if bias is None:
        bias = pair_bias(Z, ln_z_gamma, ln_z_beta, w_b)         # [H, I (query i), I (key j)]
    out = np.zeros((len(rows), I, w_o.shape[1]), dtype=np.float64)
    for r, s in enumerate(rows):
        valid = msa_mask[s]
        if valid.any():
            mh = layer_norm(Ms[s], ln_m_gamma, ln_m_beta)       # [I, c_m]
            q, k, v = _heads(mh @ w_q, H), _heads(mh @ w_k, H), _heads(mh @ w_v, H)
            g = sigmoid(mh @ w_g + b_g)
            o = np.empty_like(q)
            for h in range(H):
                o[h] = softmax_attention(q[h], k[h], v[h], bias[h], valid)
            out[r] = _gate_and_project(o, g, w_o, b_o)
            out[r][~valid] = 0.0
    if residual:
        out = np.asarray(Ms, dtype=np.float64)[list(rows)] + out
    return out
