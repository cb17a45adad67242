"""Pins for the fp64 oracle: checks against facts fixed by the mathematics, not
against the oracle's own formula.

- hand-derived worked examples (tests/golden/worked_examples.json);
- brute force on tiny inputs in 40-digit arithmetic with the naive softmax
  exp(s)/sum exp(s) (no max subtraction);
- the closed form for two keys (a logistic weighting of v0 and v1);
- an independent blockwise online-softmax recomputation: running max and
  running normaliser, earlier partial sums rescaled when a larger score arrives
  (ring-attention page, "technical insight"; deferred normalisation at the end of
  the loop, news article section 1, FlashAttention-2);
- invariants: probability rows sum to 1, constant V, equal scores, per-row
  score shifts, N = 1, causal first/last rows;
- library routines: torch's scaled_dot_product_attention in float64 and
  scipy's logsumexp;
- planted mistakes: deliberately broken copies of the oracle must fail at least
  one of the above.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle.attention import attention, attention_head, attention_probs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


def _num(x):
    if isinstance(x, (int, float)):
        return float(x)
    table = {"ln2": math.log(2), "ln3": math.log(3), "ln4": math.log(4), "ln7": math.log(7),
             "ln7/4": math.log(7 / 4), "0": 0.0, "1": 1.0, "14/3": 14 / 3}
    return table[x]


def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


# ----------------------------------------------------------------------------
# reference checks, parameterised by the implementation so that planted
# mistakes can be run through the same checks
# ----------------------------------------------------------------------------

def check_golden(fn):
    for c in _golden_cases():
        q, k, v = (np.array(c[x], dtype=np.float64) for x in ("q", "k", "v"))
        o, lse = fn(q, k, v, c["causal"], _num(c["scale"]))
        exp_o = np.array([[_num(x) for x in row] for row in c["o"]])
        exp_lse = np.array([_num(x) for x in c["lse"]])
        np.testing.assert_allclose(o, exp_o, rtol=0, atol=1e-12, err_msg=c["name"])
        np.testing.assert_allclose(lse, exp_lse, rtol=0, atol=1e-12, err_msg=c["name"])


def _bruteforce_mp(q, k, v, causal, scale):
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    N, d = q.shape
    dv = v.shape[1]
    o = np.zeros((N, dv))
    lse = np.zeros(N)
    for i in range(N):
        ws = []
        for j in range(k.shape[0]):
            if causal and j > i:
                ws.append(mpmath.mpf(0))
                continue
            s = mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(q[i, c]) * mpmath.mpf(k[j, c]) for c in range(d))
            ws.append(mpmath.e ** s)
        z = mpmath.fsum(ws)
        for c in range(dv):
            o[i, c] = float(mpmath.fsum(w * mpmath.mpf(v[j, c]) for j, w in enumerate(ws)) / z)
        lse[i] = float(mpmath.log(z))
    return o, lse


def check_bruteforce(fn, seeds=range(12)):
    for seed in seeds:
        g = np.random.default_rng(1000 + seed)
        N = int(g.integers(1, 9))
        d = int(g.integers(1, 5))
        dv = int(g.integers(1, 4))
        q, k = g.standard_normal((N, d)), g.standard_normal((N, d))
        v = g.standard_normal((N, dv))
        scale = float(g.uniform(0.2, 1.5))
        for causal in (False, True):
            o, lse = fn(q, k, v, causal, scale)
            bo, blse = _bruteforce_mp(q, k, v, causal, scale)
            np.testing.assert_allclose(o, bo, rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(lse, blse, rtol=1e-13, atol=1e-13)


def check_two_keys(fn):
    g = np.random.default_rng(7)
    for _ in range(20):
        d = 3
        q = g.standard_normal((1, d))
        k = g.standard_normal((2, d))
        v = g.standard_normal((2, 4))
        scale = 0.7
        a = scale * float(q[0] @ k[0])
        b = scale * float(q[0] @ k[1])
        sig = lambda x: 1.0 / (1.0 + math.exp(-x))  # noqa: E731
        exp_o = sig(a - b) * v[0] + sig(b - a) * v[1]
        exp_lse = max(a, b) + math.log1p(math.exp(-abs(a - b)))
        o, lse = fn(q, k, v, False, scale)
        np.testing.assert_allclose(o[0], exp_o, rtol=1e-14, atol=1e-14)
        assert abs(lse[0] - exp_lse) < 1e-14


def blockwise_online(q, k, v, causal, scale, block):
    """Independent recomputation with the online-softmax recurrence: keys are
    visited block by block keeping, per query row, a running max m, a running
    normaliser l and an unnormalised accumulator acc; whenever a block raises the
    max, the earlier l and acc are multiplied by exp(m_old - m_new).  Division by
    l happens once, after the last block."""
    N, _ = q.shape
    Nk = k.shape[0]
    m = np.full(N, -np.inf)
    l = np.zeros(N)
    acc = np.zeros((N, v.shape[1]))
    for j0 in range(0, Nk, block):
        j1 = min(Nk, j0 + block)
        s = scale * np.einsum("id,jd->ij", q, k[j0:j1])
        if causal:
            jj = np.arange(j0, j1)[None, :]
            ii = np.arange(N)[:, None]
            s = np.where(jj > ii, -np.inf, s)
        m_blk = s.max(axis=1)
        m_new = np.maximum(m, m_blk)
        alive = np.isfinite(m_new)
        corr = np.where(alive & np.isfinite(m), np.exp(np.where(alive, m - m_new, 0.0)), 0.0)
        pexp = np.where(alive[:, None], np.exp(s - np.where(alive, m_new, 0.0)[:, None]), 0.0)
        l = l * corr + pexp.sum(axis=1)
        acc = acc * corr[:, None] + pexp @ v[j0:j1]
        m = m_new
    return acc / l[:, None], m + np.log(l)


def check_blockwise(fn):
    g = np.random.default_rng(11)
    for N, d in ((1, 8), (37, 16), (200, 64), (300, 32)):
        q = g.standard_normal((N, d)) * 2.0
        k = g.standard_normal((N, d)) * 2.0
        v = g.standard_normal((N, d))
        for causal in (False, True):
            o, lse = fn(q, k, v, causal, 1 / math.sqrt(d))
            for block in (1, 7, 64, 128):
                bo, blse = blockwise_online(q, k, v, causal, 1 / math.sqrt(d), block)
                np.testing.assert_allclose(o, bo, rtol=1e-12, atol=1e-12)
                np.testing.assert_allclose(lse, blse, rtol=1e-12, atol=1e-12)


def check_invariants(fn):
    g = np.random.default_rng(5)
    N, d = 50, 8
    q, k, v = g.standard_normal((N, d)), g.standard_normal((N, d)), g.standard_normal((N, 5))
    for causal in (False, True):
        # constant V gives constant O
        o, _ = fn(q, k, np.full((N, 5), 3.25), causal, 0.9)
        np.testing.assert_allclose(o, 3.25, rtol=0, atol=1e-13)
        # equal scores (Q = 0) give the mean of the visible V rows, lse = ln(#visible)
        o, lse = fn(np.zeros((N, d)), k, v, causal, 0.9)
        for i in range(N):
            vis = i + 1 if causal else N
            np.testing.assert_allclose(o[i], v[:vis].mean(axis=0), rtol=0, atol=1e-13)
            assert abs(lse[i] - math.log(vis)) < 1e-13
        # adding c_i to every score of row i leaves O unchanged and shifts lse by c_i
        c = g.standard_normal(N) * 3
        scale = 0.9
        q2 = np.concatenate([q, (c / scale)[:, None]], axis=1)
        k2 = np.concatenate([k, np.ones((N, 1))], axis=1)
        o1, l1 = fn(q, k, v, causal, scale)
        o2, l2 = fn(q2, k2, v, causal, scale)
        np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(l2, l1 + c, rtol=1e-12, atol=1e-12)
    # N = 1: o = v0, lse = scale * q.k
    o, lse = fn(q[:1], k[:1], v[:1], False, 0.9)
    np.testing.assert_allclose(o[0], v[0], atol=1e-15)
    assert abs(lse[0] - 0.9 * float(q[0] @ k[0])) < 1e-13
    # causal row 0 is v0; causal last row equals the non-causal last row
    oc, lc = fn(q, k, v, True, 0.9)
    on, ln_ = fn(q, k, v, False, 0.9)
    np.testing.assert_allclose(oc[0], v[0], atol=1e-15)
    np.testing.assert_allclose(oc[-1], on[-1], rtol=1e-14, atol=1e-14)
    assert abs(lc[-1] - ln_[-1]) < 1e-13
    # the causal mask matters: some earlier row differs
    assert np.abs(oc[1:-1] - on[1:-1]).max() > 1e-3


def check_torch_sdpa(fn):
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(9)
    for N, d, dv in ((1, 4, 4), (17, 8, 8), (130, 32, 32), (257, 64, 16)):
        q, k, v = g.standard_normal((N, d)), g.standard_normal((N, d)), g.standard_normal((N, dv))
        for causal in (False, True):
            scale = 1 / math.sqrt(d)
            o, _ = fn(q, k, v, causal, scale)
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q)[None, None], torch.from_numpy(k)[None, None],
                torch.from_numpy(v)[None, None], is_causal=causal, scale=scale)[0, 0].numpy()
            np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)


def check_scipy_lse(fn):
    torch = pytest.importorskip("torch")
    from scipy.special import logsumexp
    g = np.random.default_rng(13)
    N, d = 90, 16
    q, k, v = g.standard_normal((N, d)) * 3, g.standard_normal((N, d)), g.standard_normal((N, d))
    for causal in (False, True):
        s = (torch.from_numpy(q) @ torch.from_numpy(k).T).numpy() * 0.5
        if causal:
            s = s + np.triu(np.full((N, N), -np.inf), 1)
        ref = logsumexp(s, axis=1)
        _, lse = fn(q, k, v, causal, 0.5)
        np.testing.assert_allclose(lse, ref, rtol=1e-13, atol=1e-13)


ALL_CHECKS = [check_golden, check_bruteforce, check_two_keys, check_blockwise, check_invariants,
              check_torch_sdpa, check_scipy_lse]


# ----------------------------------------------------------------------------
# the pins themselves
# ----------------------------------------------------------------------------

def oracle_fn(q, k, v, causal, scale):
    return attention_head(q, k, v, causal, scale)


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(oracle_fn)


def test_probability_rows_sum_to_one():
    g = np.random.default_rng(3)
    q, k = g.standard_normal((64, 16)) * 4, g.standard_normal((64, 16)) * 4
    for causal in (False, True):
        p = attention_probs(q, k, causal, 0.25)
        np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-12)
        assert (p >= 0).all()
        if causal:
            assert np.all(np.triu(p, 1) == 0)


def test_row_subset_matches_full():
    g = np.random.default_rng(4)
    q, k, v = (g.standard_normal((300, 16)) for _ in range(3))
    rows = np.array([0, 5, 128, 299])
    for causal in (False, True):
        o_full, l_full = attention_head(q, k, v, causal, 0.3)
        o_sub, l_sub = attention_head(q, k, v, causal, 0.3, rows=rows)
        np.testing.assert_allclose(o_sub, o_full[rows], rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(l_sub, l_full[rows], rtol=1e-14, atol=1e-15)


def test_batched_matches_heads():
    g = np.random.default_rng(6)
    q, k, v = (g.standard_normal((2, 3, 20, 8)) for _ in range(3))
    o, lse = attention(q, k, v, True, 0.4)
    for b in range(2):
        for h in range(3):
            oh, lh = attention_head(q[b, h], k[b, h], v[b, h], True, 0.4)
            np.testing.assert_array_equal(o[b, h], oh)
            np.testing.assert_array_equal(lse[b, h], lh)


def test_key_range_partials_merge_to_full():
    """Partial results over disjoint key ranges, merged with weights
    exp(lse_part - lse_total), reproduce the full result (the blockwise
    combination the ring-attention page describes)."""
    g = np.random.default_rng(8)
    N, d = 200, 16
    q, k, v = (g.standard_normal((N, d)) for _ in range(3))
    for causal in (False, True):
        o, lse = attention_head(q, k, v, causal, 0.25)
        cuts = [0, 33, 128, 200]
        parts = [attention_head(q, k, v, causal, 0.25, key_lo=a, key_hi=b) for a, b in zip(cuts, cuts[1:])]
        lses = np.stack([p[1] for p in parts])
        tot = np.logaddexp.reduce(lses, axis=0)
        w = np.exp(lses - tot[None])
        merged = sum(w[i][:, None] * np.nan_to_num(parts[i][0]) for i in range(len(parts)))
        np.testing.assert_allclose(tot, lse, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(merged, o, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------
# planted mistakes: each broken variant must fail at least one check
# ----------------------------------------------------------------------------

def _variant(kind):
    def fn(q, k, v, causal, scale):
        # a planted mistake may leave a row without visible keys (strict_causal):
        # its 0/0 and log(0) are the point, not a test failure
        with np.errstate(divide="ignore", invalid="ignore"):
            return _variant_body(kind, q, k, v, causal, scale)
    return fn


def _variant_body(kind, q, k, v, causal, scale):
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    N = q.shape[0]
    sc = 1.0 if kind == "no_scale" else scale
    s = sc * (q @ k.T)
    if kind == "transposed_scores":
        s = sc * (k @ q.T) if k.shape[0] == N else s.T
    if causal:
        ii = np.arange(N)[:, None]
        jj = np.arange(k.shape[0])[None, :]
        if kind == "strict_causal":
            s = np.where(jj >= ii, -np.inf, s)
        elif kind == "mask_lower":
            s = np.where(jj < ii, -np.inf, s)
        elif kind != "ignore_causal":
            s = np.where(jj > ii, -np.inf, s)
    m = s.max(axis=1)
    if kind == "strict_causal":
        m = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m[:, None])
    l = e.sum(axis=1)
    p = e / (l[:, None] if kind != "no_normalise" else 1.0)
    o = p @ (v if kind != "use_keys" else k[:, : v.shape[1]] if k.shape[1] >= v.shape[1] else v * 2)
    if kind == "drop_last_key":
        o = (e[:, :-1] / l[:, None]) @ v[:-1] if N > 1 else o
    lse = m + (np.log(l) if kind not in ("lse_base2", "lse_no_max") else
               (np.log2(l) if kind == "lse_base2" else np.log(l) - m))
    return o, lse


@pytest.mark.parametrize("kind", ["no_scale", "transposed_scores", "strict_causal", "mask_lower",
                                  "ignore_causal", "no_normalise", "use_keys", "drop_last_key",
                                  "lse_base2", "lse_no_max"])
def test_planted_mistake_is_caught(kind):
    fn = _variant(kind)
    caught = []
    for check in ALL_CHECKS:
        try:
            check(fn)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            caught.append(check.__name__)
    assert caught, f"no pin catches the planted mistake {kind!r}"


def test_variant_harness_is_faithful():
    """The unmodified variant passes every check (so a failure above is the plant)."""
    fn = _variant("none")
    for check in ALL_CHECKS:
        check(fn)
