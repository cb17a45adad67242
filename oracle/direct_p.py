"""Plain float64 CPU oracle for the Direct-P FP4 attention forward.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU leg
may call it; the library never does.  It shares no code with the CUDA sources or
with the input generator's FP4 codec (the e2m1 rounding below is its own).

The "Hardware-Aware FP4 FlashAttention-4" summary (gist.science) describes
Direct-P for non-causal inference on Blackwell's FP4 tensor cores: instead of
computing every probability exactly and then scaling and rounding it into the
4-bit format, the raw scores are mapped straight to the hardware's FP4 codes,
which removes the intermediate steps; the 4-bit P feeds the P V product.  The
summary gives no formulas.  The reading implemented here (and in the library)
uses the MXFP4 format of the P V operands -- e2m1 elements, one power-of-two
scale per 32 consecutive keys -- and takes each block's scale from the block's
largest *score*, so that a code follows from its score alone:

For one query row i with (dequantised) q_i, keys k_j and values v_j:
  1. t_ij = scale * log2(e) * (q_i . k_j)   (base-2 units); under the causal mask
     keys j > i are absent.
  2. For each block b of 32 keys (j = 32b .. 32b + 31) with a visible key:
     E_ib = ceil(max_{j in b} t_ij), an integer.
  3. code_ij = e2m1_RNE_satfinite(2^(t_ij - E_ib + 2)) and
     p_ij = value(code_ij) * 2^(E_ib - 2); absent keys have p_ij = 0.
  4. l_i = sum_j p_ij,  o_i = (sum_j p_ij v_j) / l_i,  lse_i = ln(l_i).

Since p_ij approximates 2^(t_ij) = exp(scale q_i . k_j), lse_i approximates the
exact log-sum-exp and o_i the exact attention output.  The result does not
depend on the order in which keys are visited nor on any running maximum.  The
kernel takes the code decision of step 3 in float32 (tensor-core scores, one
fused multiply-add, ex2.approx), so a value within a few float32 ulps of a
rounding boundary can land on the neighbouring code; the parity tests bound the
effect of such rare flips.
"""
from __future__ import annotations

import numpy as np

LOG2E = 1.4426950408889634
BLOCK = 32
E2M1_VALUES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def e2m1_round(x):
    """Non-negative x -> (code 0..7, value) of the nearest e2m1 magnitude; a tie
    goes to the even code (IEEE round-to-nearest-even of the 1-bit mantissa);
    values above 6 saturate to 6."""
    x = np.asarray(x, dtype=np.float64)
    vals = np.asarray(E2M1_VALUES)
    dist = np.abs(x[..., None] - vals)                       # distance to every code
    best = dist.min(axis=-1, keepdims=True)
    ties = dist == best
    codes = np.arange(8)
    # among the nearest codes prefer an even one (at most two are nearest)
    even_pick = np.where(ties & (codes % 2 == 0), codes, 99).min(axis=-1)
    any_pick = np.where(ties, codes, 99).min(axis=-1)
    code = np.where(even_pick < 99, even_pick, any_pick)
    code = np.where(x >= 6.0, 7, code)
    return code, vals[code]


def direct_p_probs(t_rows):
    """Steps 2-3 for rows of base-2 scores t [R, N] (absent keys = -inf; N a
    multiple of 32) -> (p [R, N] float64, codes [R, N] int, E [R, N/32] with
    -inf for blocks without a visible key)."""
    t = np.asarray(t_rows, dtype=np.float64)
    R, N = t.shape
    assert N % BLOCK == 0, "Direct-P blocks are 32 keys"
    tb = t.reshape(R, N // BLOCK, BLOCK)
    bmax = tb.max(axis=2)
    E = np.ceil(bmax)                                        # -inf for an empty block
    Ef = np.where(np.isfinite(E), E, 0.0)
    with np.errstate(over="ignore", invalid="ignore"):
        y = np.exp2(tb - Ef[..., None] + 2.0)                # 0 for absent keys
    code, val = e2m1_round(np.where(np.isfinite(tb), y, 0.0))
    p = val * np.exp2(Ef - 2.0)[..., None]
    p = np.where(np.isfinite(E)[..., None], p, 0.0)
    code = np.where(np.isfinite(E)[..., None], code, 0)
    return p.reshape(R, N), code.reshape(R, N), E


def direct_p_head(q, k, v, causal, scale, rows=None):
    """Direct-P attention for one head: q [Nq, d], k [N, d], v [N, dv] (float64
    values, already dequantised).  Returns (o [R, dv], lse [R]) for query
    positions `rows` (default all)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    t = (scale * LOG2E) * (q[rows] @ k.T)                   # step 1
    if causal:
        t = np.where(np.arange(k.shape[0])[None, :] > rows[:, None], -np.inf, t)
    p, _, _ = direct_p_probs(t)                              # steps 2-3
    l = p.sum(axis=1)                                        # step 4
    o = (p @ v) / l[:, None]
    return o, np.log(l)

