"""Pins for the Direct-P FP4 oracle (oracle/direct_p.py): hand-derived worked
examples, closed forms (equal scores; integer scores within three binades of
their block maximum reproduce exact softmax attention), an independent second
e2m1 rounding, invariances, and planted mistakes that each fail a pin."""
import json
import math
import os

import numpy as np
import pytest

from exact_tiled_attention_16_gb300 import synth
from oracle import direct_p as dp
from oracle.attention import attention_head

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "direct_p_examples.json")
LN2 = math.log(2.0)


def _row_inputs(ex):
    """A one-row problem whose base-2 scores are exactly the listed t: d = 1,
    q = [1], k_j = t_j, scale = ln 2 (so scale * log2(e) = 1); absent keys get a
    score 10^4 below everything (their p underflows to 0)."""
    n = ex["n_keys"]
    k = np.full((n, 1), -1e4)
    v = np.zeros((n, 1))
    for pos, t, val in ex["keys"]:
        k[pos, 0] = t
        v[pos, 0] = val
    return np.ones((1, 1)), k, v


def check_worked_examples(head=dp.direct_p_head, probs=dp.direct_p_probs):
    for ex in json.load(open(GOLDEN))["examples"]:
        q, k, v = _row_inputs(ex)
        p, _, _ = probs(k.T.copy())
        pos = [kk[0] for kk in ex["keys"]]
        np.testing.assert_allclose(p[0, pos], ex["p"], rtol=0, atol=1e-15, err_msg=ex["name"])
        o, lse = head(q, k, v, False, LN2)
        assert o[0, 0] == pytest.approx(ex["o"][0] / ex["o"][1], rel=1e-14), ex["name"]
        assert lse[0] == pytest.approx(math.log(ex["l"][0] / ex["l"][1]), rel=1e-14), ex["name"]


def check_equal_scores(head=dp.direct_p_head, probs=dp.direct_p_probs):
    """Q = 0: every score is 0, every block exponent 0, every code 4 -> p = 1:
    O is the mean of the visible V rows and lse = ln(#visible), exactly."""
    g = np.random.default_rng(0)
    N, d = 96, 8
    k, v = g.standard_normal((N, d)), g.standard_normal((N, d))
    for causal in (False, True):
        o, lse = head(np.zeros((N, d)), k, v, causal, 0.3)
        cnt = np.arange(1, N + 1) if causal else np.full(N, N)
        ref = np.cumsum(v, axis=0) / cnt[:, None] if causal else np.broadcast_to(v.mean(0), (N, d))
        np.testing.assert_allclose(o, ref, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(lse, np.log(cnt), rtol=1e-14)


def check_integer_scores(head=dp.direct_p_head, probs=dp.direct_p_probs):
    """Integer base-2 scores: 2^(t - E + 2) is a power of two, exact in e2m1 for
    t >= E - 3 (values 4, 2, 1, 0.5) and 0 for t <= E - 4 (0.25 ties to 0).  So
    (i) scores within three of their block maximum give exact softmax attention
    and (ii) lower scores are dropped -- both checked against formulas written
    here, not against the oracle."""
    g = np.random.default_rng(1)
    N, d = 64, 4
    # (i): each block's scores in {m-3..m}
    t = np.concatenate([g.integers(-3, 1, size=32) + 5, g.integers(-3, 1, size=32) - 2]).astype(float)
    q, k = np.ones((1, 1)), t[:, None]
    v = g.standard_normal((N, d))
    o, lse = head(q, k, v, False, LN2)
    ro, rl = attention_head(q, k, v, False, LN2)
    np.testing.assert_allclose(o, ro, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse, rl, rtol=1e-13)
    # (ii): one block with scores spread over ten binades
    t2 = np.zeros(32)
    t2[:] = -np.arange(32) % 10
    w = np.where(t2 >= t2.max() - 3, np.exp2(t2), 0.0)
    o2, lse2 = head(np.ones((1, 1)), t2[:, None], v[:32], False, LN2)
    np.testing.assert_allclose(o2[0], (w @ v[:32]) / w.sum(), rtol=1e-13)
    assert lse2[0] == pytest.approx(math.log(w.sum()), rel=1e-14)


def check_invariances(head=dp.direct_p_head, probs=dp.direct_p_probs):
    """Permuting keys inside a block, or permuting whole blocks, changes nothing;
    adding an integer c to every base-2 score multiplies every p by 2^c (O fixed,
    lse + c ln 2)."""
    g = np.random.default_rng(2)
    N, d = 128, 16
    q, k, v = (g.standard_normal((5, d)), g.standard_normal((N, d)), g.standard_normal((N, d)))
    o, lse = head(q, k, v, False, 0.7)
    perm = np.concatenate([g.permutation(32) + 32 * b for b in g.permutation(4)])
    o2, lse2 = head(q, k[perm], v[perm], False, 0.7)
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=1e-13)
    t = 0.7 * dp.LOG2E * (q @ k.T)
    p1, _, _ = probs(t)
    p2, _, _ = probs(t + 3.0)
    np.testing.assert_allclose(p2, p1 * 8.0, rtol=1e-14)


ALL = [check_worked_examples, check_equal_scores, check_integer_scores, check_invariances]


@pytest.mark.parametrize("check", ALL, ids=lambda c: c.__name__)
def test_direct_p_pin(check):
    check()


def test_e2m1_rounding_two_implementations_agree():
    """The oracle's nearest-value search and the input generator's codec (written
    separately from the format definition) agree on a dense grid, every tie and
    the saturation range."""
    vals = np.array(dp.E2M1_VALUES)
    mids = (vals[:-1] + vals[1:]) / 2
    grid = np.concatenate([np.linspace(0, 7, 7001), mids, vals, [6.5, 100.0]])
    code, val = dp.e2m1_round(grid)
    ref = synth.e2m1_encode_satfinite(grid)
    np.testing.assert_array_equal(code, ref)
    np.testing.assert_array_equal(val, synth.e2m1_decode(ref))
    # the ties, by the rule: even code
    np.testing.assert_array_equal(dp.e2m1_round(mids)[0], [0, 2, 2, 4, 4, 6, 6])


def test_close_to_exact_attention():
    """Direct-P is an approximation (the summary reports measurable drift and
    lower similarity): on N(0,1) inputs its rows keep a cosine similarity with
    the exact output of about 0.975 (4-bit probabilities: ~20% relative error per
    kept element, elements below 1/16 of their block's largest dropped), and lse
    stays within 0.2 of the exact value."""
    g = np.random.default_rng(3)
    N, d = 512, 64
    q, k, v = (g.standard_normal((N, d)) for _ in range(3))
    o, lse = dp.direct_p_head(q, k, v, False, 1 / 8)
    ro, rl = attention_head(q, k, v, False, 1 / 8)
    cos = (o * ro).sum(1) / np.linalg.norm(o, axis=1) / np.linalg.norm(ro, axis=1)
    assert np.median(cos) > 0.97 and cos.min() > 0.9
    assert np.abs(lse - rl).max() < 0.2


def _broken(kind):
    def probs(t_rows):
        t = np.asarray(t_rows, dtype=np.float64)
        R, N = t.shape
        tb = t.reshape(R, N // 32, 32)
        bmax = tb.max(axis=2)
        if kind == "row_exponent":
            bmax = np.broadcast_to(t.max(axis=1, keepdims=True), bmax.shape)
        E = np.floor(bmax) if kind == "floor" else np.ceil(bmax)
        off = 1.0 if kind == "offset_1" else 2.0
        Ef = np.where(np.isfinite(E), E, 0.0)
        with np.errstate(over="ignore", invalid="ignore"):
            y = np.exp2(tb - Ef[..., None] + off)
        code, val = dp.e2m1_round(np.where(np.isfinite(tb), y, 0.0))
        if kind == "ties_odd":
            vals = np.array(dp.E2M1_VALUES)
            yy = np.where(np.isfinite(tb), y, 0.0)
            tie = np.isin(yy, (vals[:-1] + vals[1:]) / 2)
            val = np.where(tie & (code % 2 == 0), vals[np.minimum(code + 1, 7)], val)
        scale = np.exp2(Ef - off)[..., None]
        p = val if kind == "no_block_scale" else val * scale
        p = np.where(np.isfinite(E)[..., None], p, 0.0)
        return p.reshape(R, N), code.reshape(R, N), E

    def head(q, k, v, causal, scale, rows=None):
        q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
        rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows)
        t = scale * dp.LOG2E * (q[rows] @ k.T)
        if causal:
            t = np.where(np.arange(k.shape[0])[None, :] > rows[:, None], -np.inf, t)
        p, _, _ = probs(t)
        l = np.exp2(t).sum(1) if kind == "exact_normaliser" else p.sum(1)
        return (p @ v) / l[:, None], np.log(l)
    return head, probs


@pytest.mark.parametrize("kind", ["floor", "offset_1", "no_block_scale", "row_exponent", "exact_normaliser",
                                  "ties_odd"])
def test_planted_mistakes_fail(kind):
    head, probs = _broken(kind)
    failed = 0
    for check in ALL:
        try:
            check(head, probs)
        except AssertionError:
            failed += 1
    assert failed > 0, kind
