"""Plain fp64 CPU oracle for the exact attention forward pass.

TEST INFRASTRUCTURE ONLY.  Nothing on the library's compute path imports this
module; it exists so that the GPU kernels can be checked against an independent,
obviously correct computation.  It shares no code with the CUDA sources.

What it computes is the plain definition of scaled dot-product attention, which
the FlashAttention pages say the tiled algorithm reproduces exactly ("no loss of
accuracy", full equivalence with standard attention: FlashAttention-2 article,
introduction and "Performance"; the ring-attention page, "technical insight":
blockwise online softmax gives a result mathematically equal to full attention).
It therefore does NOT tile: the whole score row is materialised, as in the
standard self-attention the FlashAttention-2 article describes under
"Background" (O(N^2) memory), and softmax is taken in two passes.

For one head with query rows q_i, keys k_j and values v_j (all float64):
  1. s_ij = scale * sum_c q_ic k_jc for every key j; under the causal mask
     s_ij = -inf for j > i (square, top-left aligned: key j is visible to
     query i iff j <= i, so every row sees at least key 0).
  2. m_i = max_j s_ij;  l_i = sum_j exp(s_ij - m_i).
  3. p_ij = exp(s_ij - m_i) / l_i;  o_i = sum_j p_ij v_j.
  4. lse_i = m_i + ln(l_i)   (natural log of sum_j exp(s_ij), scaled scores).

numpy's matmul serves as the dot-product step; exp and log are numpy float64.
"""
from __future__ import annotations

import numpy as np


def _scores(q, k, causal, scale, rows, key_lo=0, key_hi=None):
    """Step 1: the masked, scaled score rows s[r, j] for query positions `rows`
    against keys key_lo..key_hi-1 (absolute key positions)."""
    n_keys = k.shape[0]
    if key_hi is None:
        key_hi = n_keys
    s = scale * (q[rows, :] @ k[key_lo:key_hi, :].T)
    if causal:
        key_pos = np.arange(key_lo, key_hi)[None, :]
        s = np.where(key_pos > np.asarray(rows)[:, None], -np.inf, s)
    return s


def attention_probs(q, k, causal, scale, rows=None):
    """p[r, j]: the softmax probabilities of steps 1-3 for query rows `rows`."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    if rows is None:
        rows = np.arange(q.shape[0])
    s = _scores(q, k, causal, scale, rows)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=1, keepdims=True)


def attention_head(q, k, v, causal, scale, rows=None, key_lo=0, key_hi=None):
    """Exact attention for one head.

    q [Nq, d], k [Nk, d], v [Nk, dv] (any float type; widened to float64).
    rows: query positions to evaluate (default all).  key_lo/key_hi restrict the
    keys to a contiguous range (used for partial results over a key shard; the
    default is every key).  Returns (o [R, dv] float64, lse [R] float64).
    A row whose every key is masked gets o = 0 and lse = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if rows is None:
        rows = np.arange(q.shape[0])
    rows = np.asarray(rows, dtype=np.int64)
    if key_hi is None:
        key_hi = k.shape[0]
    s = _scores(q, k, causal, scale, rows, key_lo, key_hi)          # step 1
    m = s.max(axis=1)                                                 # step 2
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    e = np.exp(s - m_safe[:, None])
    l = e.sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        p = np.where(empty[:, None], 0.0, e / np.where(empty, 1.0, l)[:, None])  # step 3
        o = p @ v[key_lo:key_hi, :]
        lse = np.where(empty, -np.inf, m_safe + np.log(np.where(empty, 1.0, l)))  # step 4
    return o, lse


def attention(q, k, v, causal, scale):
    """Exact attention for every head of q, k, v [B, H, N, d] -> (o [B,H,N,d], lse [B,H,N])."""
    q = np.asarray(q)
    B, H, N, _ = q.shape
    dv = v.shape[-1]
    o = np.empty((B, H, N, dv), dtype=np.float64)
    lse = np.empty((B, H, N), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = attention_head(q[b, h], k[b, h], v[b, h], causal, scale)
    return o, lse
