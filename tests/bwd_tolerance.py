"""Error bounds for the BF16 attention backward against the fp64 gradient oracle.

The kernels compute scores, P, dP and every product in fp32 and round four
things to bf16 (relative error at most U = 2^-9 each): O (read back for
D_i = do_i . o_i), P^T (the A operand of dV = P^T dO), dS (the A operand of dQ
and dK) and the outputs.  A result-relative bound fails where the exact gradient
vanishes (one visible key makes dS zero), so both bounds below are taken against
the size of the terms that are summed, from the oracle's own P:

  worst case, per element (the absolute-value computation):
    a_ij = |do_i| . |v_j|,  m_ij = p_ij (a_ij + sum_j' p_ij' a_ij')
    |d dq_i| <= C_ELEM U scale sum_j m_ij |k_j|,  |d dk_j| <= C_ELEM U scale sum_i m_ij |q_i|,
    |d dv_j| <= C_ELEM U sum_i p_ij |do_i|
  aggregate (independent roundings add in quadrature):
    r_ij = p_ij (|dp_ij| + |D_i|)
    ||d dq||_F <= C_FRO U || scale sqrt(sum_j r_ij^2 k_j^2) ||_F, and likewise for dk
    (r^T, q) and dv (p^T, do).

The constants allow for the two or three roundings that reach each element with
a factor of two or more to spare.  tests/test_bwd_tolerance.py checks on the CPU
that oracle gradients rounded to bf16 pass and that planted mistakes fail.
"""
from __future__ import annotations

import numpy as np

from oracle.attention import attention_probs

U = 2.0 ** -9
C_ELEM = 8.0
C_FRO = 8.0


def _weights(p, dp, a):
    d_row = (p * dp).sum(axis=1, keepdims=True)
    m_abs = p * (a + (p * a).sum(axis=1, keepdims=True))
    m_rw = p * (np.abs(dp) + np.abs(d_row))
    return m_abs, m_rw


def bwd_bounds(q, k, v, do, causal, scale, rows=None, keys=None, row_chunk=2048):
    """Bounds for dq on query positions `rows` and dk, dv on key positions `keys`
    (default: all).  Returns {"dq"|"dk"|"dv": (worst [R|K, d], rw [R|K, d])}."""
    q, k, v, do = (np.asarray(x, np.float64) for x in (q, k, v, do))
    n = q.shape[0]
    rows = np.arange(n) if rows is None else np.asarray(rows, np.int64)
    keys = np.arange(k.shape[0]) if keys is None else np.asarray(keys, np.int64)
    aq, ak, av, ado = (np.abs(x) for x in (q, k, v, do))
    out = {}
    p = attention_probs(q, k, causal, scale, rows)
    m_abs, m_rw = _weights(p, do[rows] @ v.T, ado[rows] @ av.T)
    out["dq"] = (scale * (m_abs @ ak), scale * np.sqrt((m_rw ** 2) @ (k ** 2)))
    kw = np.zeros((keys.size, q.shape[1]))
    kr = np.zeros_like(kw)
    vw = np.zeros((keys.size, v.shape[1]))
    vr = np.zeros_like(vw)
    for r0 in range(0, n, row_chunk):
        r = np.arange(r0, min(n, r0 + row_chunk))
        p = attention_probs(q, k, causal, scale, r)
        m_abs, m_rw = _weights(p, do[r] @ v.T, ado[r] @ av.T)
        kw += scale * (m_abs[:, keys].T @ aq[r])
        kr += scale ** 2 * ((m_rw[:, keys] ** 2).T @ (q[r] ** 2))
        pk = p[:, keys]
        vw += pk.T @ ado[r]
        vr += (pk ** 2).T @ (do[r] ** 2)
    out["dk"] = (kw, np.sqrt(kr))
    out["dv"] = (vw, np.sqrt(vr))
    return out


def check(got, ref, bounds, what):
    """Raise AssertionError if got is outside the bounds around ref; returns the
    two ratios (worst elementwise, aggregate) in units of their allowances."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    worst, rw = bounds
    if not np.isfinite(got).all():
        raise AssertionError(f"{what}: non-finite values")
    diff = np.abs(got - ref)
    allow = C_ELEM * U * worst
    r_elem = float((diff / np.maximum(allow, 1e-300)).max()) if diff.size else 0.0
    fro_allow = C_FRO * U * np.linalg.norm(rw)
    r_fro = float(np.linalg.norm(diff) / max(fro_allow, 1e-300))
    if r_elem > 1.0:
        i = np.unravel_index(np.argmax(diff / np.maximum(allow, 1e-300)), diff.shape)
        raise AssertionError(f"{what}: element {i} error {diff[i]:.3e} > allowance {allow[i]:.3e}")
    if r_fro > 1.0:
        raise AssertionError(f"{what}: Frobenius error {np.linalg.norm(diff):.3e} > allowance {fro_allow:.3e}")
    return r_elem, r_fro
