"""Plain fp64 CPU oracle for the gradients of exact attention (test
infrastructure only; the library never calls it).

The forward pass is o_i = sum_j p_ij v_j with p_i = softmax_j(s_ij),
s_ij = scale * q_i . k_j (masked to -inf for j > i under the causal mask).  Given
the upstream gradient do = dL/do, the gradients are the chain rule written out
(the training use of FlashAttention-2 in the wiki article's "Performance"
section needs them; the article gives no formulas, so these are the textbook
derivatives of the definition):

  dv_j  = sum_i p_ij do_i                       (dV = P^T dO)
  dp_ij = do_i . v_j                            (dP = dO V^T)
  D_i   = sum_j p_ij dp_ij  (= do_i . o_i)
  ds_ij = p_ij (dp_ij - D_i)                    (softmax Jacobian)
  dq_i  = scale * sum_j ds_ij k_j               (dQ = scale dS K)
  dk_j  = scale * sum_i ds_ij q_i               (dK = scale dS^T Q)

P is materialised from the plain definition (oracle.attention.attention_probs);
numpy matmul serves as the dot-product step.
"""
from __future__ import annotations

import numpy as np

from .attention import attention_probs


def attention_bwd_head(q, k, v, do, causal, scale):
    """Gradients for one head: q, k, v, do [N, d] -> (dq, dk, dv) float64."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    p = attention_probs(q, k, causal, scale)
    dv = p.T @ do
    dp = do @ v.T
    d_row = (p * dp).sum(axis=1, keepdims=True)
    ds = p * (dp - d_row)
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv


def attention_bwd(q, k, v, do, causal, scale):
    """[B, H, N, d] arrays -> (dq, dk, dv) float64 of the same shape."""
    B, H = np.asarray(q).shape[:2]
    out = [np.empty(np.asarray(x).shape, np.float64) for x in (q, k, v)]
    for b in range(B):
        for h in range(H):
            dq, dk, dv = attention_bwd_head(q[b, h], k[b, h], v[b, h], do[b, h], causal, scale)
            out[0][b, h], out[1][b, h], out[2][b, h] = dq, dk, dv
    return tuple(out)


def _grad_rows(q, k, v, do, causal, scale, rows):
    """p, dp and ds for the query positions `rows` (every key), per the
    definitions above; each row depends only on its own scores."""
    p = attention_probs(q, k, causal, scale, rows)
    dp = do[rows] @ v.T
    d_row = (p * dp).sum(axis=1, keepdims=True)
    return p, p * (dp - d_row)


def attention_bwd_query_rows(q, k, v, do, causal, scale, rows):
    """dq for the query positions `rows` only -> [R, d] float64."""
    q, k, v, do = (np.asarray(x, np.float64) for x in (q, k, v, do))
    rows = np.asarray(rows, np.int64)
    _, ds = _grad_rows(q, k, v, do, causal, scale, rows)
    return scale * (ds @ k)


def attention_bwd_key_rows(q, k, v, do, causal, scale, keys, row_chunk=2048):
    """(dk, dv) for the key positions `keys` only -> two [K, d] float64 arrays.

    Column j of P needs every query row's normaliser, so every row of P and dS is
    formed (row_chunk query rows at a time, each row exactly as in
    attention_bwd_head) and only the requested columns are kept."""
    q, k, v, do = (np.asarray(x, np.float64) for x in (q, k, v, do))
    keys = np.asarray(keys, np.int64)
    n = q.shape[0]
    p_cols = np.empty((n, keys.size))
    ds_cols = np.empty((n, keys.size))
    for r0 in range(0, n, row_chunk):
        rows = np.arange(r0, min(n, r0 + row_chunk))
        p, ds = _grad_rows(q, k, v, do, causal, scale, rows)
        p_cols[rows] = p[:, keys]
        ds_cols[rows] = ds[:, keys]
    return scale * (ds_cols.T @ q), p_cols.T @ do
