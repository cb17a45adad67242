"""Pins for the fp64 gradient oracle: central finite differences of the forward
oracle, torch autograd through scaled_dot_product_attention in float64,
invariants of the softmax Jacobian, and planted mistakes."""
import numpy as np
import pytest

from oracle.attention import attention_head
from oracle.attention_bwd import attention_bwd, attention_bwd_head, attention_bwd_key_rows, attention_bwd_query_rows


def _loss(q, k, v, do, causal, scale):
    o, _ = attention_head(q, k, v, causal, scale)
    return float((o * do).sum())


def check_finite_differences(fn):
    g = np.random.default_rng(0)
    for causal in (False, True):
        N, d = 6, 3
        q, k, v, do = (g.standard_normal((N, d)) for _ in range(4))
        scale = 0.8
        dq, dk, dv = fn(q, k, v, do, causal, scale)
        h = 1e-6
        for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp = x.copy()
                xm = x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = {"q": q, "k": k, "v": v}
                args_m = {"q": q, "k": k, "v": v}
                args_p[name] = xp
                args_m[name] = xm
                num[idx] = (_loss(args_p["q"], args_p["k"], args_p["v"], do, causal, scale)
                            - _loss(args_m["q"], args_m["k"], args_m["v"], do, causal, scale)) / (2 * h)
            np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-7, err_msg=f"d{name} causal={causal}")


def check_torch_autograd(fn):
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(1)
    for N, d in ((1, 4), (33, 8), (130, 16)):
        for causal in (False, True):
            q, k, v, do = (g.standard_normal((N, d)) for _ in range(4))
            scale = 1 / np.sqrt(d)
            tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
            o = torch.nn.functional.scaled_dot_product_attention(tq[None, None], tk[None, None], tv[None, None],
                                                                 is_causal=causal, scale=scale)[0, 0]
            o.backward(torch.tensor(do))
            dq, dk, dv = fn(q, k, v, do, causal, scale)
            for a, b in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
                np.testing.assert_allclose(a, b.numpy(), rtol=1e-10, atol=1e-12)


def check_invariants(fn):
    g = np.random.default_rng(2)
    N, d = 40, 8
    q, k, v, do = (g.standard_normal((N, d)) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv = fn(q, k, v, do, causal, 0.5)
        # each row of dS sums to zero, so the key gradients sum to zero ...
        np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12)
        # ... and every row of P sums to one, so the value gradients sum to sum_i do_i
        np.testing.assert_allclose(dv.sum(axis=0), do.sum(axis=0), atol=1e-12)
        # a constant upstream gradient along V's directions gives dq = dk = 0 when V is constant
        dq2, dk2, _ = fn(q, k, np.ones((N, d)), do, causal, 0.5)
        np.testing.assert_allclose(dq2, 0.0, atol=1e-12)
        np.testing.assert_allclose(dk2, 0.0, atol=1e-12)
    # causal: the first query only sees key 0, so its dq is zero and v_0 gets do_0 in full from it
    dq, dk, dv = fn(q, k, v, do, True, 0.5)
    np.testing.assert_allclose(dq[0], 0.0, atol=1e-13)
    # the last key is seen only by the last query: dv_{N-1} = p_{N-1,N-1} do_{N-1}
    s_last = 0.5 * (q[-1] @ k.T)
    p_ll = np.exp(s_last[-1] - s_last.max()) / np.exp(s_last - s_last.max()).sum()
    np.testing.assert_allclose(dv[-1], p_ll * do[-1], rtol=1e-12, atol=1e-13)


ALL_CHECKS = [check_finite_differences, check_torch_autograd, check_invariants]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_bwd_oracle_pin(check):
    check(attention_bwd_head)


def _sampled(q, k, v, do, causal, scale):
    """The sampled-output oracle asked for every row and key (in an odd order,
    with a row chunk that splits the rows unevenly) must meet the same pins."""
    n = np.asarray(q).shape[0]
    order = np.random.default_rng(3).permutation(n)
    dq = np.empty((n, np.asarray(q).shape[1]))
    dq[order] = attention_bwd_query_rows(q, k, v, do, causal, scale, order)
    dk_s, dv_s = attention_bwd_key_rows(q, k, v, do, causal, scale, order, row_chunk=7)
    dk = np.empty_like(dq)
    dv = np.empty((n, np.asarray(v).shape[1]))
    dk[order], dv[order] = dk_s, dv_s
    return dq, dk, dv


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_sampled_bwd_oracle_pin(check):
    check(_sampled)


def _broken(kind):
    def fn(q, k, v, do, causal, scale):
        dq, dk, dv = attention_bwd_head(q, k, v, do, causal, scale)
        if kind == "dq_no_scale":
            return dq / scale, dk, dv
        if kind == "dk_transposed_role":
            return dq, dk[::-1].copy(), dv
        if kind == "dv_without_p":
            return dq, dk, np.asarray(do).copy()
        if kind == "drop_D":
            from oracle.attention import attention_probs
            p = attention_probs(q, k, causal, scale)
            ds = p * (np.asarray(do) @ np.asarray(v).T)
            return scale * ds @ k, scale * ds.T @ q, dv
        return dq, dk, dv
    return fn


@pytest.mark.parametrize("kind", ["dq_no_scale", "dk_transposed_role", "dv_without_p", "drop_D"])
def test_bwd_planted_mistake_is_caught(kind):
    caught = 0
    for check in ALL_CHECKS:
        try:
            check(_broken(kind))
        except AssertionError:
            caught += 1
    assert caught > 0


def _batched_autograd(q, k, v, do, causal, scale):
    torch = pytest.importorskip("torch")
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    o.backward(torch.tensor(do))
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


def _batched_swapped(q, k, v, do, causal, scale):
    """A planted (b, h) indexing slip: head (b, h) written to slot (h, b) of a
    transposed batch layout, then transposed back the wrong way."""
    B, H = q.shape[:2]
    out = [np.empty(x.shape, np.float64) for x in (q, k, v)]
    for b in range(B):
        for h in range(H):
            g = attention_bwd_head(q[b, h], k[b, h], v[b, h], do[b, h], causal, scale)
            bb, hh = divmod(h * B + b, H)
            for o_, x in zip(out, g):
                o_[bb, hh] = x
    return tuple(out)


@pytest.mark.parametrize("causal", [False, True])
def test_batched_bwd_matches_autograd_and_heads(causal):
    """The batched gradient oracle (the smoke check's reference) against torch
    autograd through float64 scaled_dot_product_attention on a [B, H, N, d]
    batch of distinct heads, and head by head against attention_bwd_head; a
    (b, h) indexing slip fails it (B != H, so any mix-up of heads shows)."""
    g = np.random.default_rng(9)
    B, H, N, d = 2, 3, 17, 8
    q, k, v, do = (g.standard_normal((B, H, N, d)) for _ in range(4))
    scale = 0.35
    got = attention_bwd(q, k, v, do, causal, scale)
    ref = _batched_autograd(q, k, v, do, causal, scale)
    for a, b in zip(got, ref):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12)
    for b in range(B):
        for h in range(H):
            for a, r in zip(got, attention_bwd_head(q[b, h], k[b, h], v[b, h], do[b, h], causal, scale)):
                np.testing.assert_array_equal(a[b, h], r)
    bad = _batched_swapped(q, k, v, do, causal, scale)
    assert any(not np.allclose(a, r, rtol=1e-6, atol=1e-8) for a, r in zip(bad, ref))
