"""The backward pass's tolerance (tests/bwd_tolerance.py) accepts the oracle's
gradients after bf16 rounding of their inputs' products and outputs, and rejects
planted mistakes: mistakes are planted in the oracle's output, on the CPU."""
import numpy as np
import pytest

from exact_tiled_attention_16_gb300 import synth
from oracle.attention import attention_head, attention_probs
from oracle.attention_bwd import attention_bwd_head
from tests.bwd_tolerance import bwd_bounds, check


def _bf16(x):
    return synth.bf16_bits_to_f64(synth.f32_to_bf16_bits(np.asarray(x, np.float32)))


def _case(n, d, causal, seed):
    w = synth.make_bf16(1, 1, n, d, causal, seed=seed)
    q, k, v = w.head_f64(0, 0)
    do = synth.bf16_bits_to_f64(synth.make_grad_out(1, 1, n, d, seed=seed)[0, 0])
    return q, k, v, do, w.scale


def _emulated_bf16_kernel(q, k, v, do, causal, scale):
    """The backward with the kernels' bf16 roundings applied (O for D, P^T for
    dV, dS for dQ and dK, the outputs), everything else in float64."""
    p = attention_probs(q, k, causal, scale)
    o, _ = attention_head(q, k, v, causal, scale)
    d_row = (do * _bf16(o)).sum(axis=1, keepdims=True)
    dp = do @ v.T
    ds = _bf16(p * (dp - d_row) * scale)
    return _bf16(ds @ k), _bf16(ds.T @ q), _bf16(_bf16(p).T @ do)


CASES = [(1, 64, False), (7, 128, True), (300, 64, True), (300, 128, False), (700, 64, False)]


@pytest.mark.parametrize("n,d,causal", CASES)
def test_bf16_roundings_pass(n, d, causal):
    q, k, v, do, scale = _case(n, d, causal, seed=n + d)
    ref = attention_bwd_head(q, k, v, do, causal, scale)
    got = _emulated_bf16_kernel(q, k, v, do, causal, scale)
    b = bwd_bounds(q, k, v, do, causal, scale)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        r_elem, r_fro = check(g, r, b[name], name)
        assert r_elem < 0.5 and r_fro < 0.5, (name, r_elem, r_fro)


def _planted(kind, q, k, v, do, causal, scale):
    dq, dk, dv = attention_bwd_head(q, k, v, do, causal, scale)
    p = attention_probs(q, k, causal, scale)
    if kind == "dS_without_D":
        ds = p * (do @ v.T)
        return scale * ds @ k, scale * ds.T @ q, dv
    if kind == "dq_sign":
        return -dq, dk, dv
    if kind == "dk_missing_scale":
        return dq, dk / scale, dv
    if kind == "dv_P_not_transposed":
        return dq, dk, p @ do
    if kind == "dq_key_off_by_one":
        ds = p * (do @ v.T - (p * (do @ v.T)).sum(axis=1, keepdims=True))
        return scale * ds @ np.roll(k, 1, axis=0), dk, dv
    if kind == "causal_mask_dropped":
        return attention_bwd_head(q, k, v, do, not causal, scale)
    raise ValueError(kind)


KINDS = ["dS_without_D", "dq_sign", "dk_missing_scale", "dv_P_not_transposed", "dq_key_off_by_one",
         "causal_mask_dropped"]


@pytest.mark.parametrize("kind", KINDS)
def test_planted_mistakes_fail(kind):
    q, k, v, do, scale = _case(300, 64, True, seed=11)
    ref = attention_bwd_head(q, k, v, do, True, scale)
    got = _planted(kind, q, k, v, do, True, scale)
    b = bwd_bounds(q, k, v, do, True, scale)
    failed = 0
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        try:
            check(g, r, b[name], name)
        except AssertionError:
            failed += 1
    assert failed > 0, kind


def test_sampled_bounds_match_full():
    q, k, v, do, scale = _case(300, 64, True, seed=3)
    full = bwd_bounds(q, k, v, do, True, scale)
    rows = np.array([0, 5, 127, 128, 299])
    part = bwd_bounds(q, k, v, do, True, scale, rows=rows, keys=rows, row_chunk=64)
    for name in ("dq", "dk", "dv"):
        for a, b in zip(part[name], full[name]):
            np.testing.assert_allclose(a, b[rows], rtol=1e-12, atol=1e-300)
