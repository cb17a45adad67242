"""Tolerance of the Direct-P FP4 path against its oracle (oracle/direct_p.py).

The kernel takes the same decisions as the oracle -- block exponents
E = ceil(max t) and codes e2m1(2^(t - E + 2)) -- but in float32: its scores t are
tensor-core fp32 sums of e4m3 products times an fp32 multiplier, the exponential
is ex2.approx.  Relative to the exact t that is an error of at most about
2^-21 |t| + 2^-22.  So the outputs must agree with the oracle up to

  * bf16 rounding of O (2^-9 |o|) and fp32 accumulation of P V (bounded
    generously by 2^-14 sum_j p_j |v_j| / l), and
  * the effect of any decision that lies within that reach of its boundary: a
    code whose t is within delta of a rounding midpoint of e2m1 (it may land on
    either neighbour: a change of one code step times the block scale), or a
    block whose largest t is within delta of an integer (E may differ by one:
    every code of the block may change, by at most half its value plus a quarter
    of the block scale).

For every row the allowance is the sum of these terms, so rows without a fragile
decision are held to the rounding terms alone.
"""
from __future__ import annotations

import numpy as np

from oracle import direct_p as dp

MIDPOINTS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
STEPS = np.array([0.5, 0.5, 0.5, 0.5, 1.0, 1.0, 2.0])  # gap between the codes on either side


def row_allowances(q, k, v, causal, scale, rows):
    """Oracle output and allowances for query positions `rows` of one head
    (float64 dequantised inputs).  Returns (o, lse, allow_o [R, d], allow_lse [R],
    n_fragile [R]: the number of fragile decisions of each row)."""
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    rows = np.asarray(rows, np.int64)
    t = (scale * dp.LOG2E) * (q[rows] @ k.T)
    if causal:
        t = np.where(np.arange(k.shape[0])[None, :] > rows[:, None], -np.inf, t)
    # the compared values come from the oracle itself; p and E (its steps 2-3)
    # only size the allowances below
    o, lse = dp.direct_p_head(q, k, v, causal, scale, rows=rows)
    p, _, E = dp.direct_p_probs(t)
    l = np.exp(lse)
    R, N = t.shape
    finite = np.isfinite(t)
    tmax = np.where(finite, np.abs(t), 0).max(axis=1, keepdims=True)
    delta = 2.0 ** -19 * tmax + 2.0 ** -20                     # reach of the fp32 decisions in t
    Eb = np.repeat(np.where(np.isfinite(E), E, 0.0), dp.BLOCK, axis=1)
    scale_b = np.exp2(Eb - 2.0)
    # codes near a rounding midpoint
    with np.errstate(divide="ignore", invalid="ignore"):
        t_mid = Eb[..., None] - 2.0 + np.log2(MIDPOINTS)           # [R, N, 7]
        near = finite[..., None] & (np.abs(t[..., None] - t_mid) <= delta[..., None])
    dp_code = (near * STEPS).max(axis=2) * scale_b                 # [R, N] possible change of p
    # block exponents near an integer
    bmax = np.where(finite, t, -np.inf).reshape(R, N // dp.BLOCK, dp.BLOCK).max(axis=2)
    with np.errstate(invalid="ignore"):
        near_int = np.isfinite(bmax) & (np.abs(bmax - np.round(bmax)) <= delta)
    blk = np.repeat(near_int, dp.BLOCK, axis=1)
    dp_blk = np.where(blk & finite, 0.5 * p + 0.25 * scale_b, 0.0)
    dp_any = dp_code + dp_blk
    n_fragile = (dp_any > 0).sum(axis=1)
    fragile = n_fragile > 0
    frag_o = np.zeros_like(o)
    for r in np.nonzero(fragile)[0]:
        idx = np.nonzero(dp_any[r])[0]
        frag_o[r] = (dp_any[r, idx, None] * np.abs(v[idx] - o[r])).sum(axis=0) / l[r]
    base_o = 2.0 ** -8 * np.abs(o) + 2.0 ** -14 * (p @ np.abs(v)) / l[:, None]
    allow_lse = 2.0 ** -18 * (1.0 + np.abs(lse)) + dp_any.sum(axis=1) / l
    return o, lse, base_o + 2.0 * frag_o, allow_lse, n_fragile
